// abi.cu -- library-wide entry points of libsamspec.so (version, error text)
// and the decode step that chains verification and the automata update.
#include "samspec.h"

extern "C" {

int samspec_version(void) { return 100; }  // 0.1.0

const char* samspec_strerror(int code) {
  switch (code) {
    case SAMSPEC_OK: return "ok";
    case SAMSPEC_EINVAL: return "invalid argument";
    case SAMSPEC_ESIZE: return "size outside the documented limits or workspace too small";
    case SAMSPEC_EDTYPE: return "unknown logits dtype";
    case SAMSPEC_ECUDA: return "CUDA runtime error";
    case SAMSPEC_EALIGN: return "pointer below the required alignment";
    case SAMSPEC_ST_CAPACITY: return "sequence: token, state or transition capacity exhausted";
    case SAMSPEC_ST_HASHFULL: return "sequence: transition hash full";
    case SAMSPEC_ST_TOKEN: return "sequence: token outside [0, vocab)";
    case SAMSPEC_ST_LOOPCAP: return "sequence: link walk exceeded its bound";
    case SAMSPEC_ST_BADROW: return "sequence: logits row with NaN, +inf or all -inf";
    case SAMSPEC_ST_BADDRAFT: return "sequence: draft length, draft token or n_new out of range";
    case SAMSPEC_ST_TIMEOUT: return "sequence: a bounded on-chip wait ran out";
    case SAMSPEC_ST_BADPARAM: return "sequence: temperature not > 0 and finite, or top_p not > 0";
    case SAMSPEC_ST_BOUNDS: return "sequence: an automaton index left its array (debug library)";
    default: return "unknown code";
  }
}

// One decode step: verify, then extend each sequence's automaton by what the
// step emitted (accepted drafts and the bonus or resampled token), then draft
// the next step's tokens -- "SAM投机推理：长序列强化学习训练加速利器" §1.1 (the
// D-SAM is updated as soon as verified tokens exist, then queried).  Two
// launches in stream order; the emit arrays carry the tokens between them.
int sam_spec_step(sam_batch* batch, const int32_t* d_rows, int32_t n, const void* d_target,
                  int32_t target_dtype, const int32_t* d_draft, const int32_t* d_draft_len,
                  int32_t K, int32_t V, float temperature, uint64_t seed, uint64_t step,
                  int32_t* d_accept_len, int32_t* d_out_token, int32_t* d_emit,
                  int32_t* d_emit_len, int32_t* d_status, const spec_verify_debug* dbg,
                  int32_t K_next, int32_t* d_next_draft, int32_t* d_next_draft_len,
                  int32_t* d_match_len, int32_t* d_min_endpos, void* d_workspace,
                  size_t ws_bytes, samspec_stream_t stream) {
  if (!batch || !d_emit || !d_emit_len || !d_next_draft_len) return SAMSPEC_EINVAL;
  if (K_next < 0 || K_next > 32) return SAMSPEC_ESIZE;
  if (K_next > 0 && !d_next_draft) return SAMSPEC_EINVAL;
  int rc = spec_verify(d_target, target_dtype, nullptr, SAMSPEC_F32, d_draft, d_draft_len, n, K,
                       V, temperature, seed, step, d_accept_len, d_out_token, d_emit, d_emit_len,
                       d_status, dbg, d_workspace, ws_bytes, stream);
  if (rc != SAMSPEC_OK) return rc;
  rc = sam_step_rows(batch, d_rows, n, d_emit, d_emit_len, K + 1, K_next, d_next_draft,
                     d_next_draft_len, d_match_len, d_min_endpos, stream);
  return rc;
}

}  // extern "C"
