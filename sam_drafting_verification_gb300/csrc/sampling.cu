// sampling.cu -- the cut of each target row under per-request sampling
// parameters (gogongxt.com notes "投机采样", SGLang 的实现: the target
// probabilities are softmax(l / T), then top-k renormalised, then top-p
// renormalised, before the drafts are tested).
//
// Both truncations keep a set {v : l_v >= tau} (T > 0 keeps the logits'
// order):
//   top-k (0 < k < V): tau_k = the k-th largest logit counted with
//     multiplicity (every token tied with it is kept);
//   top-p (top_p < 1): of the tokens >= tau_k, those whose mass strictly
//     above them is below top_p * Z_k (Z_k: their total mass); the cut is
//     the largest logit t whose inclusive mass from the top, M(>= t),
//     reaches top_p * Z_k;
// and tau = max(tau_k, tau_p).  The verifier then masks every logit below
// tau out of its sums, so the truncated distribution is never materialised.
//
// One CTA per row finds tau exactly by radix selection over order-preserving
// 32-bit keys of the logits (8-bit digits from the top: two levels for bf16
// rows, whose low 16 key bits are fixed by the sign, four for fp32): each
// level streams the row (from L2 after the first pass) and builds a 256-bin
// histogram of counts and masses of the keys that share the prefix chosen so
// far; one warp then scans the bins from the top for the digit where the
// running count reaches k (or the running mass reaches top_p * Z_k).  Masses
// are 2^(l log2(e)/T - R) in fixed point (units of 2^-42, R = ceil(max l
// log2(e)/T)) summed with integer atomics, so the sums are exact and the
// result does not depend on the order of the additions; lanes of a warp that
// hit the same bin are combined first (one warp reduction per distinct
// digit).  Terms below 2^-43 of the row's maximum are dropped (at V = 2^22 at
// most 2^-20 of the mass).

#include <cstdint>
#include <cstring>

#include <cuda_runtime.h>

#include "common.cuh"
#include "sampling.cuh"
#include "samspec.h"

namespace samspec {
namespace {

constexpr int kThr = 256;     // threads per CTA (one CTA per row)
constexpr int kBins = 256;    // one 8-bit digit per level
constexpr float kFix = 4398046511104.f;  // 2^42: mass units of 2^-42
constexpr int kMaxV = 1 << 22;          // keeps every mass sum below 2^64

// Order-preserving key of a logit: key(a) < key(b) iff a < b, equal iff
// a == b (-0 is folded into +0 first).
__device__ __forceinline__ uint32_t order_key(float x) {
  const uint32_t u = __float_as_uint(x + 0.f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

struct CutSmem {
  uint32_t cnt[kBins];
  unsigned long long mass[kBins];
  float red[kThr / 32];
  // result of a bin scan
  uint32_t digit;
  uint32_t above_cnt;             // keys above the prefix (all levels so far)
  unsigned long long above_mass;  // their mass
  unsigned long long bin_mass;    // mass of the chosen bin
  unsigned long long total;       // mass of every bin (first top-p level)
};

// Calls f(x, valid) for every logit of the row; every lane of the CTA makes
// the same number of calls (valid = false past the end), so f may use
// warp-wide collectives.  Rows whose byte length is a multiple of 16 are read
// in 16-byte vectors.
template <int TT, typename F>
__device__ __forceinline__ void visit_row(const unsigned char* row, int V, F&& f) {
  constexpr int ES = TT ? 2 : 4;
  constexpr int VEC = 16 / ES;
  if (((size_t)V * ES) % 16 == 0) {
    const int nvec = V / VEC;
    for (int base = 0; base < nvec; base += kThr) {
      const int i = base + (int)threadIdx.x;
      const bool ok = i < nvec;
      uint4 w = make_uint4(0u, 0u, 0u, 0u);
      if (ok) w = *reinterpret_cast<const uint4*>(row + (size_t)i * 16);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (TT) {
          f(bf16_lo(ws[q]), ok);
          f(bf16_hi(ws[q]), ok);
        } else {
          f(__uint_as_float(ws[q]), ok);
        }
      }
    }
  } else {
    for (int base = 0; base < V; base += kThr) {
      const int i = base + (int)threadIdx.x;
      const bool ok = i < V;
      float x = 0.f;
      if (ok) {
        if (TT) x = __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(row)[i] << 16);
        else x = reinterpret_cast<const float*>(row)[i];
      }
      f(x, ok);
    }
  }
}

// Adds one logit (when `in`) to bin `digit` of the histogram: the lanes of the
// warp with the same digit are combined first, one warp reduction per
// distinct digit present.
__device__ __forceinline__ void hist_add(CutSmem& sh, bool in, uint32_t digit,
                                         unsigned long long fixed, int lane) {
  unsigned todo = __ballot_sync(kFullMask, in);
  // parts of the fixed-point mass that sum without overflow over 32 lanes
  const uint32_t lo = (uint32_t)(fixed & 0x1fffffull);
  const uint32_t hi = (uint32_t)(fixed >> 21);
  while (todo) {
    const int src = __ffs(todo) - 1;
    const uint32_t d = __shfl_sync(kFullMask, digit, src);
    const bool mine = in && digit == d;
    const unsigned grp = __ballot_sync(kFullMask, mine);
    const uint32_t slo = __reduce_add_sync(kFullMask, mine ? lo : 0u);
    const uint32_t shi = __reduce_add_sync(kFullMask, mine ? hi : 0u);
    if (lane == src) {
      atomicAdd(&sh.cnt[d], (uint32_t)__popc(grp));
      atomicAdd(&sh.mass[d], ((unsigned long long)shi << 21) + slo);
    }
    todo &= ~grp;
  }
}

// Warp 0: the digit where the running sum over the bins from the top (255
// down), added to what lies above the prefix, first reaches the target: a
// count of k (BY_MASS false) or a mass (BY_MASS true; the target is
// frac * total of this histogram when from_total, else need_mass).  The bins
// above the chosen one are added to above_cnt / above_mass; the chosen bin's
// mass goes to bin_mass.  If rounding keeps the sum below the target, the
// lowest non-empty bin is taken (everything under the prefix is kept).
template <bool BY_MASS>
__device__ void scan_bins(CutSmem& sh, int lane, uint32_t k, double need_mass, bool from_total,
                          double frac) {
  uint32_t c[8];
  unsigned long long ms[8];
  uint32_t csum = 0;
  unsigned long long msum = 0;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    c[q] = sh.cnt[8 * lane + q];
    ms[q] = sh.mass[8 * lane + q];
    csum += c[q];
    msum += ms[q];
  }
  // sums over the lanes above (higher bins)
  uint32_t cs = csum;
  unsigned long long mss = msum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_down_sync(kFullMask, cs, o);
    const unsigned long long u = __shfl_down_sync(kFullMask, mss, o);
    if (lane + o < 32) {
      cs += t;
      mss += u;
    }
  }
  const uint32_t cab = cs - csum;
  const unsigned long long mab = mss - msum;
  const unsigned long long total = __shfl_sync(kFullMask, mss, 0);
  const uint32_t above_c0 = sh.above_cnt;
  const unsigned long long above_m0 = sh.above_mass;
  const double need = from_total ? frac * (double)total : need_mass;
  // walk this lane's bins downwards
  int found = -1;
  uint32_t rc = cab;
  unsigned long long rm = mab;
  uint32_t fc = 0;
  unsigned long long fm = 0;
#pragma unroll
  for (int q = 7; q >= 0; --q) {
    const bool hit = BY_MASS ? (double)(above_m0 + rm + ms[q]) >= need : above_c0 + rc + c[q] >= k;
    if (found < 0 && hit) {
      found = q;
      fc = rc;
      fm = rm;
    }
    rc += c[q];
    rm += ms[q];
  }
  unsigned hitmask = __ballot_sync(kFullMask, found >= 0);
  int src;
  if (hitmask) {
    src = 31 - __clz(hitmask);
  } else {  // the lowest non-empty bin
    found = -1;
    rc = cab;
    rm = mab;
#pragma unroll
    for (int q = 7; q >= 0; --q) {
      if (c[q] > 0) {
        found = q;
        fc = rc;
        fm = rm;
      }
      rc += c[q];
      rm += ms[q];
    }
    const unsigned ne = __ballot_sync(kFullMask, found >= 0);
    src = ne ? __ffs(ne) - 1 : 0;
    if (!ne && lane == 0) {
      found = 0;
      fc = cab;
      fm = mab;
    }
  }
  if (lane == src) {
    sh.digit = (uint32_t)(8 * lane + found);
    sh.above_cnt = above_c0 + fc;
    sh.above_mass = above_m0 + fm;
    unsigned long long bm = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (q == found) bm = ms[q];
    sh.bin_mass = bm;
    sh.total = total;
  }
}

__device__ __forceinline__ float max_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

template <int TT>
__global__ void __launch_bounds__(kThr) cut_kernel(const unsigned char* target, int32_t R, int32_t V,
                                                   const float* temp, const int32_t* top_k,
                                                   const float* top_p, float* tau) {
  constexpr int ES = TT ? 2 : 4;
  constexpr int NLEV = TT ? 2 : 4;
  __shared__ CutSmem sh;
  const float INF = __int_as_float(0x7f800000);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t row = blockIdx.x;
  const int64_t b = row / R;
  const float T = temp[b];
  const int32_t k = top_k[b];
  const float tp = top_p[b];
  if (!(T > 0.f) || !(T < INF) || !(tp > 0.f)) {
    if (threadIdx.x == 0) tau[row] = __int_as_float(0x7fc00000);
    return;
  }
  const bool use_k = k > 0 && k < V;
  const bool use_p = tp < 1.f;
  if (!use_k && !use_p) {
    if (threadIdx.x == 0) tau[row] = -INF;
    return;
  }
  const unsigned char* rp = target + (size_t)row * V * ES;
  // the row maximum (NaN-propagating)
  float m = -INF;
  visit_row<TT>(rp, V, [&](float x, bool ok) {
    if (ok) m = max_nan(m, x);
  });
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max_nan(m, __shfl_xor_sync(kFullMask, m, o));
  if (lane == 0) sh.red[warp] = m;
  __syncthreads();
  m = sh.red[0];
  for (int w = 1; w < kThr / 32; ++w) m = max_nan(m, sh.red[w]);
  if (m != m || m == INF || m == -INF) {  // the verifier refuses this row
    if (threadIdx.x == 0) tau[row] = -INF;
    return;
  }
  const float cT = (float)(1.4426950408889634 / (double)T);
  const float Rf = ceilf(m * cT);
  uint32_t min_key = 0, key_k = 0, key_p = 0;
  double zk = 0.0;  // mass of the keys >= tau_k, units 2^-42
  for (int pass = 0; pass < 2; ++pass) {
    if ((pass == 0 && !use_k) || (pass == 1 && !use_p)) continue;
    uint32_t prefix = 0;
    if (threadIdx.x == 0) {
      sh.above_cnt = 0;
      sh.above_mass = 0;
    }
    for (int lev = 0; lev < NLEV; ++lev) {
      const int shift = 24 - 8 * lev;
      const uint32_t hmask = lev == 0 ? 0u : (0xffffffffu << (shift + 8));
      for (int i = threadIdx.x; i < kBins; i += kThr) {
        sh.cnt[i] = 0;
        sh.mass[i] = 0;
      }
      __syncthreads();
      visit_row<TT>(rp, V, [&](float x, bool ok) {
        const uint32_t u = order_key(x);
        const bool in = ok && u >= min_key && (u & hmask) == (prefix & hmask);
        const float e = ex2_approx(fmaf(x, cT, -Rf));
        const unsigned long long fx = in ? __float2ull_rn(e * kFix) : 0ull;
        hist_add(sh, in, (u >> shift) & 0xffu, fx, lane);
      });
      __syncthreads();
      if (warp == 0) {
        if (pass == 0)
          scan_bins<false>(sh, lane, (uint32_t)k, 0.0, false, 0.0);
        else
          scan_bins<true>(sh, lane, 0u, (double)tp * zk, !use_k && lev == 0, (double)tp);
      }
      __syncthreads();
      prefix |= sh.digit << shift;
      if (pass == 1 && !use_k && lev == 0) zk = (double)sh.total;
    }
    // bf16 keys: the low 16 bits follow from the sign
    if (TT) prefix |= (prefix & 0x80000000u) ? 0u : 0xffffu;
    if (pass == 0) {
      key_k = prefix;
      min_key = prefix;
      zk = (double)(sh.above_mass + sh.bin_mass);
    } else {
      key_p = prefix;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) tau[row] = key_value(key_k > key_p ? key_k : key_p);
}

}  // namespace

int launch_sampling_cut(const void* target, int32_t dtype, int32_t B, int32_t R, int32_t V,
                        const float* temp, const int32_t* top_k, const float* top_p, float* tau,
                        cudaStream_t stream) {
  const int64_t rows = (int64_t)B * R;
  const auto* t = static_cast<const unsigned char*>(target);
  if (dtype == SAMSPEC_F32)
    cut_kernel<0><<<(unsigned)rows, kThr, 0, stream>>>(t, R, V, temp, top_k, top_p, tau);
  else
    cut_kernel<1><<<(unsigned)rows, kThr, 0, stream>>>(t, R, V, temp, top_k, top_p, tau);
  return cudaGetLastError() == cudaSuccess ? SAMSPEC_OK : SAMSPEC_ECUDA;
}

}  // namespace samspec

using namespace samspec;

extern "C" int spec_sampling_cut(const void* d_target, int32_t target_dtype, int32_t B, int32_t R,
                                 int32_t V, const float* d_temperature, const int32_t* d_top_k,
                                 const float* d_top_p, float* d_tau, samspec_stream_t stream) {
  if (!d_target || !d_temperature || !d_top_k || !d_top_p || !d_tau) return SAMSPEC_EINVAL;
  if (B < 1 || B > (1 << 24) || R < 1 || R > 33 || V < 1 || V > kMaxV) return SAMSPEC_ESIZE;
  if (target_dtype != SAMSPEC_F32 && target_dtype != SAMSPEC_BF16) return SAMSPEC_EDTYPE;
  if (reinterpret_cast<uintptr_t>(d_target) % 16 != 0) return SAMSPEC_EALIGN;
  return launch_sampling_cut(d_target, target_dtype, B, R, V, d_temperature, d_top_k, d_top_p,
                             d_tau, reinterpret_cast<cudaStream_t>(stream));
}
