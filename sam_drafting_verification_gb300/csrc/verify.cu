// verify.cu -- lossless verification of K drafts per sequence over [B, K+1, V]
// logits, one persistent CTA per SM.
//
// Method (pages named by title and section):
//   greedy (T = 0): gogongxt.com notes "投机采样", 贪婪采样 -- keep the drafts
//     equal to the target's most probable token, emit that token at the first
//     mismatch;
//   rejection sampling (T > 0): nxbn.cn speculative-sampling article §2.2 --
//     accept draft j with probability min(1, p_target/p_draft), on rejection
//     resample from the positive part of p_target - p_draft, K+1 distributions;
//     "SAM投机推理：长序列强化学习训练加速利器" §1.1 -- eps <= alpha(x) accepts;
//     gogongxt notes, SGLang 的实现 -- p = softmax(logits / temperature), one
//     coin per draft and one for the final sample; N-gram 的特殊情况 -- model-free
//     drafts carry draft_probs = 0, so q is the indicator of the draft token and
//     the bonus sample is drawn from the target distribution itself.
//
// GB300 design.  A row of V = 151936 logits is 304-608 KB, so verification is
// a streaming reduction bound by HBM.  Each CTA owns whole sequences and walks
// their accept chains itself, so rows after the first rejection are never read
// and no inter-CTA merge is needed:
//   warp 16 (producer) issues 1-D bulk copies (cp.async.bulk, the TMA engine)
//       of 32 KB vocab tiles of the rows its sequence slots ask for into a
//       ring of shared-memory stages, completion counted on mbarriers;
//   warps 0-15 (consumers) each reduce a 1/16 slice ("warp slice") of every
//       tile from shared memory (16-byte vector reads) to a record -- the
//       slice's max and sum of 2^((l - max) log2(e)/T), or its (max, first
//       argmax) -- and release the stage;
//   warp 17 (control) claims sequences from a global counter into four slots,
//       merges the warp-slice records of a finished row in fp64, draws the
//       Philox coins, decides accept/reject and posts the next row; after the
//       final row it resamples: the slice records give the mass of every warp
//       slice, so it finds the slice holding u' * sum(r) and scans just that
//       2-8 KB slice, read again from L2, in ascending token order.
// Four slots keep the producer streaming while the control warp decides.
// Every wait is bounded by a global-timer deadline; a CTA that runs out of
// time marks its sequences SAMSPEC_ST_TIMEOUT, lets its copies in flight land
// and exits.

#include <cstdint>
#include <cstring>

#include <cuda_runtime.h>

#include "common.cuh"
#include "philox.cuh"
#include "samspec.h"

namespace samspec {
namespace {

constexpr int kCW = 16;              // consumer warps
constexpr int kProdWarp = kCW;       // producer warp
constexpr int kCtrlWarp = kCW + 1;   // control warp
constexpr int kThreads = (kCW + 2) * 32;
constexpr int kStageBytes = 32768;
constexpr int kMaxStages = 6;
constexpr int kMinStages = 3;
constexpr int kSlots = 4;
constexpr int kMaxChunks = 64;
constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s per wait

enum Kind : int32_t { kStats = 0, kResid = 1, kExit = 3 };
enum State : int32_t { kEmpty = 0, kReady = 1, kIssued = 2, kDone = 3 };

struct VParams {
  const unsigned char* target;
  const unsigned char* draftl;
  const int32_t* draft;
  const int32_t* draft_len;
  int32_t B, K, V;
  float T, cT;  // cT = log2(e) / T
  double Td;
  uint64_t seed, step;
  int32_t* accept_len;
  int32_t* out_token;
  int32_t* emit;
  int32_t* emit_len;
  int32_t* status;
  spec_verify_debug dbg;
  uint32_t* ws;  // [0] claim counter, [1] CTA exit counter, [2] error bits
  int32_t NC, NS;
  int32_t direct;  // 1: plain loads instead of bulk copies (unaligned rows)
};

struct Tag {
  int32_t slot, kind, chunk, nel, elem0, has_draft, b, j;
};

struct Slot {
  int32_t state;  // State, accessed with volatile loads/stores
  int32_t kind;   // kind of the current job (kStats: row j; kResid: row L)
  int32_t b, j, nb, L;
  int32_t cnt;    // warp records received for the current job
  int32_t smode;  // residual pass: 1 -> max(0, p - q) in units of p;
                  //                0 -> p in units of exp(x - m)
  float lmax, gmax, invZ, invZg;
};

struct Smem {
  Slot slot[kSlots];
  Tag tag[kMaxStages];
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  int32_t stage_parity[kMaxStages];  // parity of the last issue per stage
  int32_t ctrl_done;
  int32_t abort;
  int32_t prod_idle;  // the producer has issued every posted job
};

__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// NaN-propagating maxima
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}
__device__ __forceinline__ uint32_t bf16x2_max_nan(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// ---- element access ---------------------------------------------------------
// A "vector" holds VEC consecutive logits of one array: 16 bytes, or 8 bytes
// for the bf16 array of a mixed fp32/bf16 pair (so that both arrays share one
// element-to-lane map).
template <int ES, int VEC>
struct Vec {
  static constexpr int kWords = ES * VEC / 4;
  uint32_t w[kWords];
  __device__ __forceinline__ float at(int k) const {
    if (ES == 4) return __uint_as_float(w[k]);
    return (k & 1) ? bf16_hi(w[k >> 1]) : bf16_lo(w[k >> 1]);
  }
  __device__ __forceinline__ void load16(const unsigned char* p) {
    if (kWords == 4) {
      const uint4 v = *reinterpret_cast<const uint4*>(p);
      w[0] = v.x; w[1] = v.y; w[2 % kWords] = v.z; w[3 % kWords] = v.w;
    } else {
      const uint2 v = *reinterpret_cast<const uint2*>(p);
      w[0] = v.x; w[1 % kWords] = v.y;
    }
  }
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int q = 0; q < kWords; ++q) w[q] = 0;
  }
  // element-wise global loads for rows without 16-byte alignment; elements at
  // or beyond `valid` are not read (set to 0)
  __device__ __forceinline__ void load_elems(const unsigned char* p, int valid) {
    zero();
#pragma unroll
    for (int k = 0; k < VEC; ++k) {
      if (k < valid) {
        if (ES == 4) {
          w[k] = __ldg(reinterpret_cast<const uint32_t*>(p) + k);
        } else {
          const uint32_t h = __ldg(reinterpret_cast<const unsigned short*>(p) + k);
          w[k >> 1] |= (k & 1) ? (h << 16) : h;
        }
      }
    }
  }
  // NaN-propagating maximum of the vector's elements
  __device__ __forceinline__ float vmax() const {
    if (ES == 4) {
      float m = __uint_as_float(w[0]);
#pragma unroll
      for (int k = 1; k < VEC; ++k) m = fmax_nan(m, __uint_as_float(w[k]));
      return m;
    }
    uint32_t a = w[0];
#pragma unroll
    for (int q = 1; q < kWords; ++q) a = bf16x2_max_nan(a, w[q]);
    return fmax_nan(bf16_lo(a), bf16_hi(a));
  }
};

template <int TT, int DT>
struct Cfg {
  static constexpr int ST = TT ? 2 : 4;
  static constexpr int SD = DT < 0 ? 0 : (DT ? 2 : 4);
  static constexpr int MAXS = ST > SD ? ST : SD;
  static constexpr int VEC = 16 / MAXS;
  static constexpr int E_TILE = DT < 0 ? kStageBytes / ST : (ST == SD ? kStageBytes / (2 * ST) : 4096);
  static constexpr int SL = E_TILE / kCW;        // elements per warp slice
  static constexpr int VPL = SL / (32 * VEC);    // vectors per lane per array
  static constexpr int DOFF = E_TILE * ST;       // byte offset of the draft part
  static_assert(VPL >= 1 && VPL * 32 * VEC * kCW == E_TILE, "tile shape");
  static_assert(E_TILE * (ST + SD) <= kStageBytes, "stage size");
};

template <int TT, int DT>
struct Slice {
  using C = Cfg<TT, DT>;
  Vec<C::ST, C::VEC> t[C::VPL];
  Vec<(C::SD ? C::SD : 4), C::VEC> d[(DT >= 0) ? C::VPL : 1];
};

// Loads warp slice `w` of a staged tile (bulk-copy mode) or of the tile's
// global rows (direct mode).  The draft part is read only when the tile
// carries one.
template <int TT, int DT>
__device__ __forceinline__ void load_slice_tile(Slice<TT, DT>& s, const VParams& P,
                                                const unsigned char* stage, const Tag& tg, int w,
                                                int lane) {
  using C = Cfg<TT, DT>;
#pragma unroll
  for (int i = 0; i < C::VPL; ++i) {
    const int e = w * C::SL + (i * 32 + lane) * C::VEC;  // element index in the tile
    if (!P.direct) {
      s.t[i].load16(stage + (size_t)e * C::ST);
      if (DT >= 0 && tg.has_draft) s.d[i].load16(stage + C::DOFF + (size_t)e * C::SD);
    } else {
      const int valid = tg.nel - e;
      const size_t rt = ((size_t)tg.b * (P.K + 1) + tg.j) * (size_t)P.V + tg.elem0 + e;
      s.t[i].load_elems(P.target + rt * C::ST, valid);
      if (DT >= 0 && tg.has_draft) {
        const size_t rd = ((size_t)tg.b * P.K + tg.j) * (size_t)P.V + tg.elem0 + e;
        s.d[i].load_elems(P.draftl + rd * C::SD, valid);
      }
    }
  }
}

// Loads warp slice `w` of tile `c` of row L of sequence b straight from global
// memory (the control warp's resample scan).  Returns the slice's element count.
template <int TT, int DT>
__device__ __forceinline__ int load_slice_global(Slice<TT, DT>& s, const VParams& P, int b, int L,
                                                 int c, int w, bool with_draft, int lane) {
  using C = Cfg<TT, DT>;
  const int s0 = c * C::E_TILE + w * C::SL;
  const size_t rt = ((size_t)b * (P.K + 1) + L) * (size_t)P.V;
  const size_t rd = ((size_t)b * P.K + L) * (size_t)P.V;
#pragma unroll
  for (int i = 0; i < C::VPL; ++i) {
    const int e = s0 + (i * 32 + lane) * C::VEC;  // vocab index
    const int valid = P.V - e;
    if (!P.direct) {
      // aligned rows hold whole vectors: a vector is either in range or not
      if (valid > 0) {
        s.t[i].load16(P.target + (rt + e) * C::ST);
        if (DT >= 0 && with_draft) s.d[i].load16(P.draftl + (rd + e) * C::SD);
      } else {
        s.t[i].zero();
        if (DT >= 0) s.d[i].zero();
      }
    } else {
      s.t[i].load_elems(P.target + (rt + e) * C::ST, valid);
      if (DT >= 0) {
        if (with_draft) s.d[i].load_elems(P.draftl + (rd + e) * C::SD, valid);
        else s.d[i].zero();
      }
    }
  }
  const int n = P.V - s0;
  return n < 0 ? 0 : (n > C::SL ? C::SL : n);
}

// ---- per-warp reductions over a slice ----------------------------------------
// NaN-propagating lane maximum of one array over the valid elements
template <int TT, int DT, bool FULL, bool DRAFT_ARRAY>
__device__ __forceinline__ float lane_max(const Slice<TT, DT>& s, int w, int lane, int nel) {
  using C = Cfg<TT, DT>;
  float m = -__int_as_float(0x7f800000);
#pragma unroll
  for (int i = 0; i < C::VPL; ++i) {
    if (FULL) {
      m = fmax_nan(m, DRAFT_ARRAY ? s.d[i].vmax() : s.t[i].vmax());
    } else {
      const int e = w * C::SL + (i * 32 + lane) * C::VEC;
#pragma unroll
      for (int k = 0; k < C::VEC; ++k)
        if (e + k < nel) m = fmax_nan(m, DRAFT_ARRAY ? s.d[i].at(k) : s.t[i].at(k));
    }
  }
  return m;
}

// greedy record: {max, first index of the max, NaN seen}
template <int TT, int DT, bool FULL>
__device__ __forceinline__ float4 reduce_greedy(const Slice<TT, DT>& s, int w, int lane, int nel,
                                                int elem0) {
  using C = Cfg<TT, DT>;
  const float ml = lane_max<TT, DT, FULL, false>(s, w, lane, nel);
  if (__any_sync(kFullMask, ml != ml)) return make_float4(0.f, __int_as_float(0x7fffffff), 1.f, 0.f);
  const float M = warp_max(ml);
  int32_t idx = 0x7fffffff;
  if (ml == M) {  // only the lanes holding the maximum look for its first position
#pragma unroll
    for (int i = 0; i < C::VPL; ++i) {
      const int e = w * C::SL + (i * 32 + lane) * C::VEC;
#pragma unroll
      for (int k = 0; k < C::VEC; ++k)
        if ((FULL || e + k < nel) && s.t[i].at(k) == M && idx == 0x7fffffff) idx = elem0 + e + k;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) idx = min(idx, __shfl_xor_sync(kFullMask, idx, o));
  return make_float4(M, __int_as_float(idx), 0.f, 0.f);
}

// {max, sum_x 2^((x - max) * cT)} of one array; NaN in the slice -> {NaN, NaN}
template <int TT, int DT, bool FULL, bool DRAFT_ARRAY>
__device__ __forceinline__ float2 reduce_softmax(const Slice<TT, DT>& s, int w, int lane, int nel,
                                                 float cT) {
  using C = Cfg<TT, DT>;
  const float NEG_INF = -__int_as_float(0x7f800000);
  const float ml = lane_max<TT, DT, FULL, DRAFT_ARRAY>(s, w, lane, nel);
  if (__any_sync(kFullMask, ml != ml))
    return make_float2(__int_as_float(0x7fc00000), __int_as_float(0x7fc00000));
  const float m = warp_max(ml);
  float z = 0.f;
  if (m != NEG_INF) {
    float part[C::VPL];
#pragma unroll
    for (int i = 0; i < C::VPL; ++i) {
      const int e = w * C::SL + (i * 32 + lane) * C::VEC;
      float v[C::VEC];
#pragma unroll
      for (int k = 0; k < C::VEC; ++k) {
        const float x = DRAFT_ARRAY ? s.d[i].at(k) : s.t[i].at(k);
        v[k] = (FULL || e + k < nel) ? ex2_approx((x - m) * cT) : 0.f;
      }
#pragma unroll
      for (int h = C::VEC / 2; h >= 1; h >>= 1)
#pragma unroll
        for (int k = 0; k < h; ++k) v[k] += v[k + h];
      part[i] = v[0];
    }
#pragma unroll
    for (int h = C::VPL / 2; h >= 1; h >>= 1)
#pragma unroll
      for (int i = 0; i < h; ++i) part[i] += part[i + h];
    z = warp_sum(part[0]);
  }
  return make_float2(m, z);
}

// residual-pass record: sum of r over the slice (fast exponential)
template <int TT, int DT, bool FULL>
__device__ __forceinline__ float reduce_resid(const Slice<TT, DT>& s, int w, int lane, int nel,
                                              const Slot& S, float cT) {
  using C = Cfg<TT, DT>;
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < C::VPL; ++i) {
    const int e = w * C::SL + (i * 32 + lane) * C::VEC;
    float part = 0.f;
#pragma unroll
    for (int k = 0; k < C::VEC; ++k) {
      if (FULL || e + k < nel) {
        const float pe = ex2_approx((s.t[i].at(k) - S.lmax) * cT);
        if (S.smode == 0) {
          part += pe;
        } else {
          float g = 0.f;
          if (DT >= 0) g = s.d[i].at(k);
          const float qe = ex2_approx((g - S.gmax) * cT);
          part += fmaxf(0.f, pe * S.invZ - qe * S.invZg);
        }
      }
    }
    acc += part;
  }
  return warp_sum(acc);
}

// residual weight of one element with the accurate exponential (resample scan)
template <int TT, int DT>
__device__ __forceinline__ float resid_elem(const Slice<TT, DT>& s, int i, int k, int vocab,
                                            int smode, int excl, float lmax, float gmax,
                                            float invZ, float invZg, float cT) {
  const float pe = exp2f((s.t[i].at(k) - lmax) * cT);
  if (smode == 0) return vocab == excl ? 0.f : pe;
  float g = 0.f;
  if (DT >= 0) g = s.d[i].at(k);
  const float qe = exp2f((g - gmax) * cT);
  return fmaxf(0.f, pe * invZ - qe * invZg);
}

// ---- outputs ---------------------------------------------------------------
__device__ void write_result(const VParams& P, int b, int L, int out, int st) {
  P.accept_len[b] = st ? -1 : L;
  P.out_token[b] = st ? -1 : out;
  if (P.status) P.status[b] = st;
  if (P.emit_len) P.emit_len[b] = st ? 0 : L + 1;
  if (P.emit) {
    for (int t = 0; t <= P.K; ++t) {
      int v = -1;
      if (!st) v = t < L ? P.draft[(size_t)b * P.K + t] : (t == L ? out : -1);
      P.emit[(size_t)b * (P.K + 1) + t] = v;
    }
  }
}

__device__ __forceinline__ float load_logit(const unsigned char* base, int es, size_t idx) {
  if (es == 4) return __ldg(reinterpret_cast<const float*>(base) + idx);
  return __uint_as_float((uint32_t)__ldg(reinterpret_cast<const unsigned short*>(base) + idx) << 16);
}

// First lane in [0, n) whose inclusive running sum of v exceeds t, or -1;
// *before receives the running sum ahead of that lane.
__device__ __forceinline__ int warp_find(double v, double t, int n, int lane, double* before) {
  const double x = lane < n ? v : 0.0;
  const double incl = warp_incl_scan_d(x, lane);
  const unsigned hit = __ballot_sync(kFullMask, lane < n && incl > t);
  if (!hit) return -1;
  const int src = __ffs(hit) - 1;
  *before = __shfl_sync(kFullMask, incl, src) - __shfl_sync(kFullMask, x, src);
  return src;
}

// ---- control warp ------------------------------------------------------------
template <int TT, int DT, bool GREEDY>
struct Control {
  using C = Cfg<TT, DT>;
  const VParams& P;
  Smem& sm;
  const float4* rec;  // [kSlots][NC][kCW]
  int lane;
  bool more;

  __device__ Control(const VParams& p, Smem& s, const float4* r, int l)
      : P(p), sm(s), rec(r), lane(l), more(true) {}

  __device__ const float4& R(int si, int c, int w) const {
    return rec[((size_t)si * P.NC + c) * kCW + w];
  }

  __device__ void finish(int b, int L, int out, int st) {
    if (lane == 0) write_result(P, b, L, out, st);
    __syncwarp();
  }

  __device__ void post(int si, int kind, int j) {
    Slot& S = sm.slot[si];
    if (lane == 0) {
      S.kind = kind;
      S.j = j;
      S.cnt = 0;
      __threadfence_block();
      vstore(&S.state, kReady);
    }
    __syncwarp();
  }

  __device__ void release(int si) {
    if (lane == 0) vstore(&sm.slot[si].state, kEmpty);
    __syncwarp();
  }

  // Claims sequences until one with valid drafts lands in slot si (or none
  // are left: the slot becomes empty).
  __device__ void refill(int si) {
    Slot& S = sm.slot[si];
    while (more) {
      uint32_t b = 0;
      if (lane == 0) b = atomicAdd(&P.ws[0], 1u);
      b = __shfl_sync(kFullMask, b, 0);
      if (b >= (uint32_t)P.B) {
        more = false;
        break;
      }
      const int nb = P.draft_len ? P.draft_len[b] : P.K;
      bool bad = nb < 0 || nb > P.K;
      if (!bad && lane < nb) {
        const int32_t d = P.draft[(size_t)b * P.K + lane];
        bad = d < 0 || d >= P.V;
      }
      if (__any_sync(kFullMask, bad)) {
        finish((int)b, -1, -1, SAMSPEC_ST_BADDRAFT);
        continue;
      }
      if (lane == 0) {
        S.b = (int32_t)b;
        S.nb = nb;
        S.L = 0;
      }
      post(si, kStats, 0);
      return;
    }
    if (lane == 0) vstore(&S.state, kEmpty);
    __syncwarp();
  }

  // Resample scan of warp slice (c, w) of row L: the first token whose running
  // residual exceeds t (ascending token id), with the accurate exponential.
  __device__ int slice_scan(int b, int L, int c, int w, double t, int smode, int excl, float lmax,
                            float gmax, float invZ, float invZg) {
    Slice<TT, DT> sl;
    const bool with_draft = DT >= 0 && smode == 1;
    const int n = load_slice_global<TT, DT>(sl, P, b, L, c, w, with_draft, lane);
    const int s0 = c * C::E_TILE + w * C::SL;
    int token = -1, last_pos = -1;
    double tt = t;
#pragma unroll
    for (int i = 0; i < C::VPL; ++i) {
      const int e = (i * 32 + lane) * C::VEC;  // index inside the slice
      float r[C::VEC];
      double s_l = 0.0;
#pragma unroll
      for (int k = 0; k < C::VEC; ++k) {
        r[k] = (e + k < n) ? resid_elem<TT, DT>(sl, i, k, s0 + e + k, smode, excl, lmax, gmax,
                                                invZ, invZg, P.cT)
                           : 0.f;
        s_l += (double)r[k];
        if (r[k] > 0.f) last_pos = s0 + e + k;
      }
      const double li = warp_incl_scan_d(s_l, lane);
      const double row_total = __shfl_sync(kFullMask, li, 31);
      if (token < 0 && row_total > tt) {
        const unsigned h2 = __ballot_sync(kFullMask, li > tt);
        const int ls = __ffs(h2) - 1;
        const double tl = tt - (__shfl_sync(kFullMask, li, ls) - __shfl_sync(kFullMask, s_l, ls));
        int found = -1;
        if (lane == ls) {
          double acc = 0.0;
          int lastk = -1;
          for (int k = 0; k < C::VEC; ++k) {
            acc += (double)r[k];
            if (r[k] > 0.f) lastk = k;
            if (acc > tl) {
              found = k;
              break;
            }
          }
          if (found < 0) found = lastk;
          if (found >= 0) found = s0 + e + found;
        }
        found = __shfl_sync(kFullMask, found, ls);
        if (found >= 0) token = found;
      }
      if (token < 0) tt -= row_total;
    }
    if (token < 0) {  // rounding put t past the slice: its last positive entry
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
        last_pos = max(last_pos, __shfl_xor_sync(kFullMask, last_pos, o));
      token = last_pos >= 0 ? last_pos : s0;
    }
    return token;
  }

  // Picks the warp slice holding t from per-tile masses (cm, two per lane:
  // tiles lane and lane + 32) and the per-slice masses of the chosen tile,
  // then scans it.
  template <typename SliceMass>
  __device__ int resample(int b, int L, double t, const double* cm, SliceMass slice_mass,
                          int smode, int excl, float lmax, float gmax, float invZ, float invZg) {
    const int NC = P.NC;
    int cstar = -1;
    double base = 0.0, before = 0.0;
    for (int q = 0; q < 2 && q * 32 < NC; ++q) {
      const int f = warp_find(cm[q], t - base, NC - q * 32, lane, &before);
      if (f >= 0) {
        cstar = q * 32 + f;
        before += base;
        break;
      }
      base += warp_sum_d((q * 32 + lane) < NC ? cm[q] : 0.0);
    }
    double tc;
    if (cstar < 0) {  // rounding left the total at or below t: last tile with mass
      int lastc = 0;
      for (int q = 0; q < 2 && q * 32 < NC; ++q) {
        const unsigned pos = __ballot_sync(kFullMask, (q * 32 + lane) < NC && cm[q] > 0.0);
        if (pos) lastc = q * 32 + 31 - __clz(pos);
      }
      cstar = lastc;
      tc = 1e300;
    } else {
      tc = t - before;
    }
    const double sm_w = lane < kCW ? slice_mass(cstar, lane) : 0.0;
    double bw = 0.0;
    int wstar = warp_find(sm_w, tc, kCW, lane, &bw);
    double tw;
    if (wstar < 0) {
      const unsigned pos = __ballot_sync(kFullMask, lane < kCW && sm_w > 0.0);
      wstar = pos ? 31 - __clz(pos) : 0;
      tw = 1e300;
    } else {
      tw = tc - bw;
    }
    return slice_scan(b, L, cstar, wstar, tw, smode, excl, lmax, gmax, invZ, invZg);
  }

  __device__ void handle(int si) {
    Slot& S = sm.slot[si];
    const int b = S.b, j = S.j, nb = S.nb;
    const int NC = P.NC;
    const size_t ro = (size_t)b * (P.K + 1) + j;

    if (GREEDY) {
      float best = -__int_as_float(0x7f800000);
      int32_t bi = 0x7fffffff;
      bool nan = false;
      for (int c = lane; c < NC; c += 32)
        for (int w = 0; w < kCW; ++w) {
          const float4 r = R(si, c, w);
          const int32_t ri = __float_as_int(r.y);
          nan |= r.z != 0.f;
          if (r.x > best || (r.x == best && ri < bi)) {
            best = r.x;
            bi = ri;
          }
        }
      warp_argmax(best, bi);
      nan = __any_sync(kFullMask, nan);
      const bool bad = nan || bi == 0x7fffffff || best == -__int_as_float(0x7f800000);
      if (lane == 0) {
        if (P.dbg.row_m) P.dbg.row_m[ro] = best;
        if (P.dbg.row_arg) P.dbg.row_arg[ro] = bad ? -1 : bi;
      }
      if (bad) {
        finish(b, -1, -1, SAMSPEC_ST_BADROW);
        release(si);
        return;
      }
      if (j < nb && P.draft[(size_t)b * P.K + j] == bi) {
        post(si, kStats, j + 1);
        return;
      }
      finish(b, j, bi, 0);
      release(si);
      return;
    }

    if (S.kind == kStats) {
      // --- temperature-softmax statistics of row j ---
      float lm = -__int_as_float(0x7f800000), gm = lm;
      for (int c = lane; c < NC; c += 32)
        for (int w = 0; w < kCW; ++w) {
          const float4 r = R(si, c, w);
          lm = fmaxf(lm, r.x);
          if (DT >= 0) gm = fmaxf(gm, r.z);
        }
      lm = warp_max(lm);
      if (DT >= 0) gm = warp_max(gm);
      const float cT = P.cT;
      // slice mass in units of exp(x - lm); a NaN slice keeps its NaN
      auto mass_of = [&](const float4& r) -> double {
        return r.y == 0.f ? 0.0 : (double)r.y * (double)exp2f((r.x - lm) * cT);
      };
      double cm[2] = {0.0, 0.0};
      double zt = 0.0, zg = 0.0;
      for (int c = lane, q = 0; c < NC; c += 32, ++q) {
        double m = 0.0, g = 0.0;
        for (int w = 0; w < kCW; ++w) {
          const float4 r = R(si, c, w);
          m += mass_of(r);
          if (DT >= 0 && r.w != 0.f) g += (double)r.w * (double)exp2f((r.z - gm) * cT);
        }
        if (q < 2) cm[q] = m;
        zt += m;
        zg += g;
      }
      zt = warp_sum_d(zt);
      if (DT >= 0) zg = warp_sum_d(zg);
      const float NEG_INF = -__int_as_float(0x7f800000);
      const bool bad_t = !(lm > NEG_INF) || isinf(lm) || !isfinite(zt) || !(zt > 0.0);
      const bool bad_g = DT >= 0 && j < nb &&
                         (!(gm > NEG_INF) || isinf(gm) || !isfinite(zg) || !(zg > 0.0));
      if (lane == 0) {
        if (P.dbg.row_m) P.dbg.row_m[ro] = lm / P.T;
        if (P.dbg.row_z) P.dbg.row_z[ro] = (float)zt;
      }
      if (bad_t || bad_g) {
        finish(b, -1, -1, SAMSPEC_ST_BADROW);
        release(si);
        return;
      }
      float ua, ur;
      verify_coins(P.seed, P.step, (uint32_t)b, (uint32_t)j, &ua, &ur);
      int32_t d = -1;
      double ed = 0.0;
      if (j < nb) {
        d = P.draft[(size_t)b * P.K + j];
        const float ld = load_logit(P.target, C::ST, ro * P.V + d);
        ed = exp(((double)ld - (double)lm) / P.Td);
        const double pd = ed / zt;
        double qd = 1.0;
        if (DT >= 0) {
          const float gd = load_logit(P.draftl, C::SD, ((size_t)b * P.K + j) * P.V + d);
          qd = exp(((double)gd - (double)gm) / P.Td) / zg;
        }
        if (lane == 0) {
          if (P.dbg.p_d) P.dbg.p_d[ro] = (float)pd;
          if (P.dbg.q_d) P.dbg.q_d[ro] = (float)qd;
        }
        // accept iff u * q(d) <= p(d)  (eps <= alpha(x) with alpha = min(1, p/q))
        if ((double)ua * qd <= pd) {
          post(si, kStats, j + 1);
          return;
        }
      }
      // j is the final row L: rejected (j < nb) or the bonus row (j == nb)
      if (DT >= 0 && j < nb) {
        // residual max(0, p - q) needs both rows' full statistics: one more pass
        if (lane == 0) {
          S.L = j;
          S.lmax = lm;
          S.gmax = gm;
          S.invZ = (float)(1.0 / zt);
          S.invZg = (float)(1.0 / zg);
          S.smode = 1;
        }
        post(si, kResid, j);
        return;
      }
      // one-hot rejection: r = p without the rejected token; bonus: r = p.
      // Units: exp(x - m); the row's Z is their total.
      int excl = -1;
      double sum_r = zt;
      int cd = -1, wd = -1;
      if (j < nb && zt - ed > 0.0) {
        excl = d;
        sum_r = zt - ed;
        cd = d / C::E_TILE;
        wd = (d - cd * C::E_TILE) / C::SL;
        if ((cd & 31) == lane && (cd >> 5) < 2) {
          const double nm = cm[cd >> 5] - ed;
          cm[cd >> 5] = nm > 0.0 ? nm : 0.0;
        }
      }
      if (lane == 0 && P.dbg.res_mass) P.dbg.res_mass[b] = (float)(sum_r / zt);
      const double t = (double)ur * sum_r;
      auto slice_mass = [&](int c, int w) -> double {
        double m = mass_of(R(si, c, w));
        if (c == cd && w == wd) m = m - ed > 0.0 ? m - ed : 0.0;
        return m;
      };
      const int out = resample(b, j, t, cm, slice_mass, 0, excl, lm, gm, 0.f, 0.f);
      finish(b, j, out, 0);
      release(si);
      return;
    }

    // kResid: per-slice residual masses of row L from the second pass
    const int L = S.L;
    double cm[2] = {0.0, 0.0};
    double tot = 0.0;
    for (int c = lane, q = 0; c < NC; c += 32, ++q) {
      double m = 0.0;
      for (int w = 0; w < kCW; ++w) m += (double)R(si, c, w).x;
      if (q < 2) cm[q] = m;
      tot += m;
    }
    tot = warp_sum_d(tot);
    if (S.smode == 1 && (!(tot > 0.0) || !isfinite(tot))) {
      // zero residual (impossible in exact arithmetic): sample p instead
      if (lane == 0) S.smode = 0;
      post(si, kResid, L);
      return;
    }
    float ua, ur;
    verify_coins(P.seed, P.step, (uint32_t)b, (uint32_t)L, &ua, &ur);
    if (lane == 0 && P.dbg.res_mass) P.dbg.res_mass[b] = (float)(S.smode ? tot : 1.0);
    const double t = (double)ur * tot;
    auto slice_mass = [&](int c, int w) -> double { return (double)R(si, c, w).x; };
    const int out =
        resample(b, L, t, cm, slice_mass, S.smode, -1, S.lmax, S.gmax, S.invZ, S.invZg);
    finish(b, L, out, 0);
    release(si);
  }
};

template <int TT, int DT, bool GREEDY>
__global__ void __launch_bounds__(kThreads, 1) verify_kernel(const VParams P) {
  using C = Cfg<TT, DT>;
  extern __shared__ __align__(1024) unsigned char dsm[];
  Smem& sm = *reinterpret_cast<Smem*>(dsm);
  const size_t rec_off = (sizeof(Smem) + 15) & ~(size_t)15;
  float4* rec = reinterpret_cast<float4*>(dsm + rec_off);
  const size_t rec_bytes = (size_t)kSlots * P.NC * kCW * sizeof(float4);
  unsigned char* stages = dsm + ((rec_off + rec_bytes + 1023) & ~(size_t)1023);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int NS = P.NS;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kCW);
      sm.stage_parity[s] = -1;
    }
    for (int s = 0; s < kSlots; ++s) {
      sm.slot[s].state = kEmpty;
      sm.slot[s].cnt = 0;
    }
    sm.ctrl_done = 0;
    sm.abort = 0;
    sm.prod_idle = 0;
    mbar_fence_init();
  }
  __syncthreads();

  if (warp < kCW) {
    // ------------------------------ consumers ------------------------------
    int cs = 0;
    uint32_t cph = 0;
    for (;;) {
      const uint64_t t0 = gtimer();
      bool ok = true;
      while (!mbar_try_wait(&sm.full[cs], cph)) {
        if (vload(&sm.abort) || gtimer() - t0 > kWaitNs) {
          ok = false;
          break;
        }
      }
      if (!ok) {
        if (lane == 0) vstore(&sm.abort, 1);
        break;
      }
      const Tag tg = sm.tag[cs];
      if (tg.kind == kExit) break;
      Slot& S = sm.slot[tg.slot];
      const unsigned char* stage = stages + (size_t)cs * kStageBytes;
      Slice<TT, DT> sl;
      load_slice_tile<TT, DT>(sl, P, stage, tg, warp, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[cs]);
      const bool full = tg.nel == C::E_TILE;
      float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
      if (tg.kind == kStats) {
        if (GREEDY) {
          r = full ? reduce_greedy<TT, DT, true>(sl, warp, lane, tg.nel, tg.elem0)
                   : reduce_greedy<TT, DT, false>(sl, warp, lane, tg.nel, tg.elem0);
        } else {
          const float2 a = full ? reduce_softmax<TT, DT, true, false>(sl, warp, lane, tg.nel, P.cT)
                                : reduce_softmax<TT, DT, false, false>(sl, warp, lane, tg.nel, P.cT);
          r.x = a.x;
          r.y = a.y;
          if (DT >= 0 && tg.has_draft) {
            const float2 g = full ? reduce_softmax<TT, DT, true, true>(sl, warp, lane, tg.nel, P.cT)
                                  : reduce_softmax<TT, DT, false, true>(sl, warp, lane, tg.nel, P.cT);
            r.z = g.x;
            r.w = g.y;
          }
        }
      } else {  // kResid
        r.x = full ? reduce_resid<TT, DT, true>(sl, warp, lane, tg.nel, S, P.cT)
                   : reduce_resid<TT, DT, false>(sl, warp, lane, tg.nel, S, P.cT);
      }
      if (lane == 0) {
        rec[((size_t)tg.slot * P.NC + tg.chunk) * kCW + warp] = r;
        __threadfence_block();
        const int old = atomicAdd(&S.cnt, 1);
        if (old == P.NC * kCW - 1) {
          S.cnt = 0;
          __threadfence_block();
          vstore(&S.state, kDone);
        }
      }
      __syncwarp();
      if (++cs == NS) {
        cs = 0;
        cph ^= 1;
      }
    }
  } else if (warp == kProdWarp) {
    // ------------------------------- producer ------------------------------
    if (lane == 0) {
      int ps = 0;
      uint32_t pph = 0;
      int rr = 0;
      uint64_t t_idle = gtimer();
      for (;;) {
        if (vload(&sm.abort)) break;
        int si = -1;
        for (int k = 0; k < kSlots && si < 0; ++k) {
          const int s = (rr + k) % kSlots;
          if (vload(&sm.slot[s].state) == kReady) si = s;
        }
        if (si < 0) {
          vstore(&sm.prod_idle, 1);
          if (vload(&sm.ctrl_done)) break;
          if (gtimer() - t_idle > kWaitNs) {
            vstore(&sm.abort, 1);
            break;
          }
          __nanosleep(32);
          continue;
        }
        rr = si + 1;
        vstore(&sm.prod_idle, 0);
        __threadfence_block();
        Slot& S = sm.slot[si];
        vstore(&S.state, kIssued);
        const int kind = S.kind, b = S.b, j = S.j;
        // the draft model's row is read for rows with a draft (j < n_b): its
        // statistics, and the residual pass
        const bool with_draft =
            DT >= 0 && ((kind == kStats && j < S.nb) || (kind == kResid && S.smode == 1));
        bool ok = true;
        for (int c = 0; c < P.NC && ok; ++c) {
          const uint64_t t0 = gtimer();
          while (!mbar_try_wait(&sm.empty[ps], pph ^ 1)) {
            if (vload(&sm.abort) || gtimer() - t0 > kWaitNs) {
              ok = false;
              break;
            }
          }
          if (!ok) break;
          const int elem0 = c * C::E_TILE;
          const int nel = min(C::E_TILE, P.V - elem0);
          Tag& tg = sm.tag[ps];
          tg.slot = si;
          tg.kind = kind;
          tg.chunk = c;
          tg.nel = nel;
          tg.elem0 = elem0;
          tg.has_draft = with_draft ? 1 : 0;
          tg.b = b;
          tg.j = j;
          unsigned char* dst = stages + (size_t)ps * kStageBytes;
          if (P.direct) {
            mbar_arrive(&sm.full[ps]);
          } else {
            const size_t rt = ((size_t)b * (P.K + 1) + j) * (size_t)P.V + elem0;
            const uint32_t bt = (uint32_t)nel * C::ST;
            const uint32_t bd = with_draft ? (uint32_t)nel * C::SD : 0u;
            mbar_arrive_expect_tx(&sm.full[ps], bt + bd);
            bulk_g2s(dst, P.target + rt * C::ST, bt, &sm.full[ps]);
            if (with_draft) {
              const size_t rd = ((size_t)b * P.K + j) * (size_t)P.V + elem0;
              bulk_g2s(dst + C::DOFF, P.draftl + rd * C::SD, bd, &sm.full[ps]);
            }
          }
          sm.stage_parity[ps] = (int32_t)pph;
          if (++ps == NS) {
            ps = 0;
            pph ^= 1;
          }
        }
        if (!ok) {
          vstore(&sm.abort, 1);
          break;
        }
        t_idle = gtimer();
      }
      if (!vload(&sm.abort)) {
        // tell the consumers to stop
        const uint64_t t0 = gtimer();
        bool ok = true;
        while (!mbar_try_wait(&sm.empty[ps], pph ^ 1)) {
          if (gtimer() - t0 > kWaitNs) {
            ok = false;
            break;
          }
        }
        if (ok) {
          sm.tag[ps].kind = kExit;
          __threadfence_block();
          mbar_arrive(&sm.full[ps]);
        } else {
          vstore(&sm.abort, 1);
        }
      }
      if (vload(&sm.abort)) {
        atomicOr(&P.ws[2], 1u);
        // let every bulk copy this CTA issued land before the CTA exits
        for (int s = 0; s < NS; ++s) {
          if (sm.stage_parity[s] < 0) continue;
          const uint64_t t0 = gtimer();
          while (!mbar_try_wait(&sm.full[s], (uint32_t)sm.stage_parity[s]))
            if (gtimer() - t0 > kWaitNs) break;
        }
      }
    }
  } else if (warp == kCtrlWarp) {
    // -------------------------------- control -------------------------------
    // One sequence per CTA to begin with; another is claimed only once the
    // producer has issued everything posted (its ring still holds up to NS
    // tiles, which covers the claim), so small batches spread over all CTAs
    // and large ones keep every producer busy.
    Control<TT, DT, GREEDY> ctl(P, sm, rec, lane);
    ctl.refill(0);
    uint64_t t_idle = gtimer();
    for (;;) {
      int si = -1, free_slot = -1, ready = 0;
      if (lane == 0)
        for (int s = 0; s < kSlots; ++s) {
          const int st = vload(&sm.slot[s].state);
          if (st == kDone && si < 0) si = s;
          if (st == kEmpty && free_slot < 0) free_slot = s;
          ready += st == kReady;
        }
      si = __shfl_sync(kFullMask, si, 0);
      free_slot = __shfl_sync(kFullMask, free_slot, 0);
      ready = __shfl_sync(kFullMask, ready, 0);
      if (si >= 0) {
        __threadfence_block();
        ctl.handle(si);
        t_idle = gtimer();
        continue;
      }
      if (ctl.more && ready == 0 && free_slot >= 0 && vload(&sm.prod_idle)) {
        ctl.refill(free_slot);
        t_idle = gtimer();
        continue;
      }
      int stop = 0;
      if (lane == 0) {
        if (vload(&sm.abort)) {
          stop = 1;
        } else {
          bool all_empty = true;
          for (int s = 0; s < kSlots; ++s) all_empty &= vload(&sm.slot[s].state) == kEmpty;
          if (all_empty && !ctl.more) {
            vstore(&sm.ctrl_done, 1);
            stop = 1;
          } else if (gtimer() - t_idle > kWaitNs) {
            vstore(&sm.abort, 1);
            stop = 1;
          }
        }
      }
      stop = __shfl_sync(kFullMask, stop, 0);
      if (stop) break;
      __nanosleep(32);
    }
    if (vload(&sm.abort) && lane == 0) {
      // sequences held by this CTA's slots, and any nobody will claim now
      for (int s = 0; s < kSlots; ++s)
        if (sm.slot[s].state != kEmpty) write_result(P, sm.slot[s].b, -1, -1, SAMSPEC_ST_TIMEOUT);
      for (uint32_t b = atomicAdd(&P.ws[0], 1u); b < (uint32_t)P.B; b = atomicAdd(&P.ws[0], 1u))
        write_result(P, (int)b, -1, -1, SAMSPEC_ST_TIMEOUT);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(&P.ws[1], 1u) == gridDim.x - 1) {
      // last CTA out: reset the counters for the next launch on this workspace
      P.ws[0] = 0;
      P.ws[1] = 0;
      __threadfence();
    }
  }
}

__global__ void uniforms_kernel(int32_t B, int32_t K, uint64_t seed, uint64_t step, float* u) {
  const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (i >= (int64_t)B * (K + 1)) return;
  const int b = (int)(i / (K + 1)), j = (int)(i % (K + 1));
  verify_coins(seed, step, (uint32_t)b, (uint32_t)j, &u[2 * i], &u[2 * i + 1]);
}

// ---- host launch --------------------------------------------------------------
template <int TT, int DT, bool GREEDY>
int launch(const VParams& P0, cudaStream_t stream) {
  using C = Cfg<TT, DT>;
  VParams P = P0;
  P.NC = (P.V + C::E_TILE - 1) / C::E_TILE;
  if (P.NC > kMaxChunks) return SAMSPEC_ESIZE;
  const size_t rec_off = (sizeof(Smem) + 15) & ~(size_t)15;
  const size_t head =
      (rec_off + (size_t)kSlots * P.NC * kCW * sizeof(float4) + 1023) & ~(size_t)1023;
  // Device properties and the kernel's shared-memory opt-in are set up once per
  // device, so that later launches make no runtime calls besides the launch
  // itself (safe inside stream capture).
  constexpr int kMaxDev = 64;
  static int max_smem[kMaxDev] = {0}, sms[kMaxDev] = {0};
  static bool attr_done[kMaxDev] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return SAMSPEC_ECUDA;
  if (sms[dev] == 0) {
    if (cudaDeviceGetAttribute(&max_smem[dev], cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return SAMSPEC_ECUDA;
  }
  if (!attr_done[dev]) {
    if (cudaFuncSetAttribute(verify_kernel<TT, DT, GREEDY>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem[dev]) !=
        cudaSuccess)
      return SAMSPEC_ECUDA;
    attr_done[dev] = true;
  }
  int ns = (int)(((size_t)max_smem[dev] - head) / kStageBytes);
  if (ns > kMaxStages) ns = kMaxStages;
  if (ns < kMinStages) return SAMSPEC_ESIZE;
  P.NS = ns;
  const size_t smem = head + (size_t)ns * kStageBytes;
  const int grid = P.B < sms[dev] ? P.B : sms[dev];
  verify_kernel<TT, DT, GREEDY><<<grid, kThreads, smem, stream>>>(P);
  return cudaGetLastError() == cudaSuccess ? SAMSPEC_OK : SAMSPEC_ECUDA;
}

template <bool GREEDY>
int dispatch(const VParams& P, int tdt, int ddt, cudaStream_t stream) {
  if (GREEDY || ddt < 0) {
    return tdt == SAMSPEC_F32 ? launch<0, -1, GREEDY>(P, stream) : launch<1, -1, GREEDY>(P, stream);
  }
  if (tdt == SAMSPEC_F32)
    return ddt == SAMSPEC_F32 ? launch<0, 0, GREEDY>(P, stream) : launch<0, 1, GREEDY>(P, stream);
  return ddt == SAMSPEC_F32 ? launch<1, 0, GREEDY>(P, stream) : launch<1, 1, GREEDY>(P, stream);
}

}  // namespace
}  // namespace samspec

using namespace samspec;

extern "C" {

size_t spec_verify_workspace_bytes(int32_t B, int32_t K, int32_t V) {
  if (B < 1 || K < 1 || V < 1) return 0;
  return 256;
}

int spec_verify_workspace_init(void* d_workspace, size_t ws_bytes, samspec_stream_t stream) {
  if (!d_workspace || ws_bytes < 256) return SAMSPEC_EINVAL;
  return cudaMemsetAsync(d_workspace, 0, 256, reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? SAMSPEC_OK
             : SAMSPEC_ECUDA;
}

int spec_verify(const void* d_target, int32_t target_dtype, const void* d_draft_logits,
                int32_t draft_dtype, const int32_t* d_draft, const int32_t* d_draft_len,
                int32_t B, int32_t K, int32_t V, float temperature, uint64_t seed, uint64_t step,
                int32_t* d_accept_len, int32_t* d_out_token, int32_t* d_emit, int32_t* d_emit_len,
                int32_t* d_status, const spec_verify_debug* dbg, void* d_workspace,
                size_t ws_bytes, samspec_stream_t stream) {
  if (!d_target || !d_draft || !d_accept_len || !d_out_token || !d_workspace) return SAMSPEC_EINVAL;
  if (B < 1 || B > (1 << 24) || K < 1 || K > 32 || V < 1 || V > (1 << 24)) return SAMSPEC_ESIZE;
  if (!(temperature >= 0.f) || temperature != temperature || temperature == __builtin_inff())
    return SAMSPEC_EINVAL;
  if (target_dtype != SAMSPEC_F32 && target_dtype != SAMSPEC_BF16) return SAMSPEC_EDTYPE;
  const bool greedy = temperature == 0.f;
  int ddt = -1;
  if (d_draft_logits && !greedy) {
    if (draft_dtype != SAMSPEC_F32 && draft_dtype != SAMSPEC_BF16) return SAMSPEC_EDTYPE;
    ddt = draft_dtype;
  }
  if (ws_bytes < spec_verify_workspace_bytes(B, K, V)) return SAMSPEC_ESIZE;
  if (reinterpret_cast<uintptr_t>(d_workspace) % 256 != 0) return SAMSPEC_EALIGN;
  const int st = target_dtype == SAMSPEC_F32 ? 4 : 2;
  const int sd = ddt < 0 ? 0 : (ddt == SAMSPEC_F32 ? 4 : 2);
  if (reinterpret_cast<uintptr_t>(d_target) % 16 != 0) return SAMSPEC_EALIGN;
  if (ddt >= 0 && reinterpret_cast<uintptr_t>(d_draft_logits) % 16 != 0) return SAMSPEC_EALIGN;
  VParams P;
  std::memset(&P, 0, sizeof(P));
  P.target = static_cast<const unsigned char*>(d_target);
  P.draftl = static_cast<const unsigned char*>(d_draft_logits);
  P.draft = d_draft;
  P.draft_len = d_draft_len;
  P.B = B;
  P.K = K;
  P.V = V;
  P.T = temperature;
  P.Td = (double)temperature;
  P.cT = greedy ? 0.f : (float)(1.4426950408889634 / (double)temperature);
  P.seed = seed;
  P.step = step;
  P.accept_len = d_accept_len;
  P.out_token = d_out_token;
  P.emit = d_emit;
  P.emit_len = d_emit_len;
  P.status = d_status;
  if (dbg) P.dbg = *dbg;
  P.ws = static_cast<uint32_t*>(d_workspace);
  P.direct = ((size_t)V * st) % 16 != 0 || (sd && ((size_t)V * sd) % 16 != 0);
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return greedy ? dispatch<true>(P, target_dtype, ddt, s)
                : dispatch<false>(P, target_dtype, ddt, s);
}

int spec_uniforms(int32_t B, int32_t K, uint64_t seed, uint64_t step, float* d_u,
                  samspec_stream_t stream) {
  if (!d_u || B < 1 || K < 0 || K > 32) return SAMSPEC_EINVAL;
  const int64_t n = (int64_t)B * (K + 1);
  uniforms_kernel<<<(unsigned)((n + 255) / 256), 256, 0,
                    reinterpret_cast<cudaStream_t>(stream)>>>(B, K, seed, step, d_u);
  return cudaGetLastError() == cudaSuccess ? SAMSPEC_OK : SAMSPEC_ECUDA;
}

}  // extern "C"
