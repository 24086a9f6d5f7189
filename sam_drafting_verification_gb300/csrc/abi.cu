// abi.cu -- library-wide entry points of libsamspec.so (version, error text).
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
    default: return "unknown code";
  }
}

}  // extern "C"
