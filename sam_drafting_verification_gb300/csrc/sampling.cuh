// sampling.cuh -- internal interface of the per-request sampling-parameter
// cut (sampling.cu), used by the verification entry point in verify.cu.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

namespace samspec {

// For each of the B * R rows of target ([B, R, V], dtype SAMSPEC_F32 or
// SAMSPEC_BF16), the smallest logit kept by the temperature / top-k / top-p
// truncation of its sequence's parameters (temp, top_k, top_p: [B]) into
// tau [B, R]: -inf keeps every token (no truncation, or a row the verifier
// refuses anyway), NaN marks invalid parameters.  One launch on `stream`.
int launch_sampling_cut(const void* target, int32_t dtype, int32_t B, int32_t R, int32_t V,
                        const float* temp, const int32_t* top_k, const float* top_p, float* tau,
                        cudaStream_t stream);

}  // namespace samspec
