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
// a streaming reduction bound by HBM.  Each CTA owns whole sequences (claimed
// from a global counter) and walks their accept chains itself, so rows after
// the first rejection are never read and no inter-CTA merge is needed:
//   warp 16 (producer) claims sequences and issues 1-D bulk copies
//       (cp.async.bulk, the TMA engine) of 32 KB vocab tiles into a ring of
//       shared-memory stages, completion counted on mbarriers;
//   warps 0-15 (consumers) each reduce a 1/16 slice of every tile from shared
//       memory (16-byte vector reads) to a per-warp record -- max and sum of
//       2^((l - max) log2(e)/T) with warp shuffles, or (max, argmax) -- and
//       release the stage;
//   warp 17 (control) merges the NC tile records of a finished row in fp64,
//       draws the Philox coins, takes the accept/reject decision and posts the
//       sequence's next job (next row, residual pass, or the one-tile CDF
//       search), and writes the outputs.
// Two sequence slots per CTA keep the producer streaming one sequence while
// the other waits for its decision.  The resample needs only one tile: the
// per-tile masses of the rejected row come from its statistics pass, so the
// control warp finds the tile holding u' * sum(r) and a single tile is fetched
// again (usually from L2) for the final scan.  Every wait is bounded by a
// global-timer deadline; a CTA that runs out of time marks its sequences
// SAMSPEC_ST_TIMEOUT, lets its copies in flight land and exits.

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
constexpr int kSlots = 2;
constexpr int kMaxChunks = 64;
constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s per wait

enum Kind : int32_t { kStats = 0, kResid = 1, kSearch = 2, kExit = 3, kInvalid = 4 };
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
  int32_t kind;   // kind of the current job
  int32_t b, j, nb, L;
  int32_t c0, c1;          // tiles [c0, c1) of the current job
  int32_t cnt;             // warp records received for the current job
  int32_t search_stage;    // stage holding the search tile (kept until scanned)
  int32_t excl;            // token whose mass is removed (one-hot rejection), or -1
  int32_t smode;           // 0: r in units of exp(x - m) (one-hot); 1: r = max(0, p - q)
  float lmax, gmax, invZ, invZg;
  double t_local;          // search target inside the chosen tile
  double zrow;             // Z of the final row
  double sum_r;            // residual mass, in the units of smode
};

__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
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
  __device__ __forceinline__ void load_smem(const unsigned char* p) {
    if (kWords == 4) {
      const uint4 v = *reinterpret_cast<const uint4*>(p);
      w[0] = v.x; w[1] = v.y; w[2 % kWords] = v.z; w[3 % kWords] = v.w;
    } else {
      const uint2 v = *reinterpret_cast<const uint2*>(p);
      w[0] = v.x; w[1 % kWords] = v.y;
    }
  }
  // element-wise global loads for rows without 16-byte alignment; elements at
  // or beyond `valid` are not read (set to 0)
  __device__ __forceinline__ void load_global(const unsigned char* p, int valid) {
#pragma unroll
    for (int q = 0; q < kWords; ++q) w[q] = 0;
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

// Loads warp slice `w` of a tile for lane `lane` from the stage (bulk-copy
// mode) or from global memory (direct mode).
// The draft part is read only when the tile carries one (tg.has_draft).
template <int TT, int DT>
__device__ __forceinline__ void load_slice(Slice<TT, DT>& s, const VParams& P,
                                           const unsigned char* stage, const Tag& tg, int w,
                                           int lane) {
  using C = Cfg<TT, DT>;
#pragma unroll
  for (int i = 0; i < C::VPL; ++i) {
    const int e = w * C::SL + (i * 32 + lane) * C::VEC;  // element index in the tile
    if (!P.direct) {
      s.t[i].load_smem(stage + (size_t)e * C::ST);
      if (DT >= 0 && tg.has_draft) s.d[i].load_smem(stage + C::DOFF + (size_t)e * C::SD);
    } else {
      const int valid = tg.nel - e;
      const size_t row_t = ((size_t)tg.b * (P.K + 1) + tg.j) * (size_t)P.V + tg.elem0 + e;
      s.t[i].load_global(P.target + row_t * C::ST, valid);
      if (DT >= 0 && tg.has_draft) {
        const size_t row_d = ((size_t)tg.b * P.K + tg.j) * (size_t)P.V + tg.elem0 + e;
        s.d[i].load_global(P.draftl + row_d * C::SD, valid);
      }
    }
  }
}

// ---- per-warp reductions over a slice ----------------------------------------
template <int TT, int DT, bool FULL>
__device__ __forceinline__ float4 reduce_greedy(const Slice<TT, DT>& s, int w, int lane, int nel,
                                                int elem0) {
  using C = Cfg<TT, DT>;
  float best = -__int_as_float(0x7f800000);
  int32_t bi = 0x7fffffff;
  bool nan = false;
#pragma unroll
  for (int i = 0; i < C::VPL; ++i) {
    const int e = w * C::SL + (i * 32 + lane) * C::VEC;
#pragma unroll
    for (int k = 0; k < C::VEC; ++k) {
      if (FULL || e + k < nel) {
        const float x = s.t[i].at(k);
        nan |= (x != x);
        if (x > best) {
          best = x;
          bi = elem0 + e + k;
        }
      }
    }
  }
  warp_argmax(best, bi);
  const bool any_nan = __any_sync(kFullMask, nan);
  return make_float4(best, __int_as_float(bi), any_nan ? 1.f : 0.f, 0.f);
}

// max and sum_x 2^((x - max) * cT) of one array of the slice
template <int TT, int DT, bool FULL, bool DRAFT_ARRAY>
__device__ __forceinline__ float2 reduce_softmax(const Slice<TT, DT>& s, int w, int lane, int nel,
                                                 float cT) {
  using C = Cfg<TT, DT>;
  const float NEG_INF = -__int_as_float(0x7f800000);
  float m = NEG_INF;
#pragma unroll
  for (int i = 0; i < C::VPL; ++i) {
    const int e = w * C::SL + (i * 32 + lane) * C::VEC;
#pragma unroll
    for (int k = 0; k < C::VEC; ++k)
      if (FULL || e + k < nel) m = fmaxf(m, DRAFT_ARRAY ? s.d[i].at(k) : s.t[i].at(k));
  }
  m = warp_max(m);
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
      // pairwise sum of the vector
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

// residual weight of one element (accurate exp2f: used where a CDF is read)
template <int TT, int DT>
__device__ __forceinline__ float resid_elem(const Slice<TT, DT>& s, int i, int k, int vocab,
                                            const Slot& S, float cT) {
  const float x = s.t[i].at(k);
  const float pe = exp2f((x - S.lmax) * cT);
  if (S.smode == 0) return vocab == S.excl ? 0.f : pe;
  float g = 0.f;
  if (DT >= 0) g = s.d[i].at(k);
  const float qe = exp2f((g - S.gmax) * cT);
  return fmaxf(0.f, pe * S.invZ - qe * S.invZg);
}

// residual weight with the fast exponential (statistics pass of the draft model's
// residual mass)
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
        float g = 0.f;
        if (DT >= 0) g = s.d[i].at(k);
        const float qe = ex2_approx((g - S.gmax) * cT);
        part += fmaxf(0.f, pe * S.invZ - qe * S.invZg);
      }
    }
    acc += part;
  }
  return warp_sum(acc);
}

template <int TT, int DT, bool FULL>
__device__ __forceinline__ float reduce_search(const Slice<TT, DT>& s, int w, int lane, int nel,
                                               int elem0, const Slot& S, float cT) {
  using C = Cfg<TT, DT>;
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < C::VPL; ++i) {
    const int e = w * C::SL + (i * 32 + lane) * C::VEC;
#pragma unroll
    for (int k = 0; k < C::VEC; ++k)
      if (FULL || e + k < nel) acc += resid_elem<TT, DT>(s, i, k, elem0 + e + k, S, cT);
  }
  return warp_sum(acc);
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

struct Smem {
  Slot slot[kSlots];
  Tag tag[kMaxStages];
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  int32_t prod_done;
  int32_t abort;
  int32_t stage_parity[kMaxStages];  // parity of the last issue per stage
  double cmass[kSlots][kMaxChunks];  // tile masses of the last statistics row
  float4 rec[kSlots][kMaxChunks][kCW];
};

// ---- control warp: merge a finished job and decide --------------------------
template <int TT, int DT, bool GREEDY>
__device__ void control_handle(const VParams& P, Smem& sm, unsigned char* stages, int si,
                               int lane) {
  using C = Cfg<TT, DT>;
  Slot& S = sm.slot[si];
  const int b = S.b;
  const double NEG_INF = -__longlong_as_double(0x7ff0000000000000ll);

  auto finish = [&](int L, int out, int st) {
    if (lane == 0) write_result(P, b, L, out, st);
    __syncwarp();
    __threadfence_block();
    if (lane == 0) vstore(&S.state, kEmpty);
    __syncwarp();
  };
  auto post = [&](int kind, int j, int c0, int c1) {
    if (lane == 0) {
      S.kind = kind;
      S.j = j;
      S.c0 = c0;
      S.c1 = c1;
      S.cnt = 0;
      __threadfence_block();
      vstore(&S.state, kReady);
    }
    __syncwarp();
  };

  if (S.kind == kInvalid) {
    finish(-1, -1, SAMSPEC_ST_BADDRAFT);
    return;
  }
  const int j = S.j;
  const int NC = P.NC;

  if (S.kind == kStats && GREEDY) {
    float best = -__int_as_float(0x7f800000);
    int32_t bi = 0x7fffffff;
    bool nan = false;
    for (int c = lane; c < NC; c += 32)
      for (int w = 0; w < kCW; ++w) {
        const float4 r = sm.rec[si][c][w];
        const int32_t ri = __float_as_int(r.y);
        nan |= r.z != 0.f;
        if (r.x > best || (r.x == best && ri < bi)) {
          best = r.x;
          bi = ri;
        }
      }
    warp_argmax(best, bi);
    nan = __any_sync(kFullMask, nan);
    const size_t ro = (size_t)b * (P.K + 1) + j;
    if (lane == 0) {
      if (P.dbg.row_m) P.dbg.row_m[ro] = best;
      if (P.dbg.row_arg) P.dbg.row_arg[ro] = (nan || bi == 0x7fffffff) ? -1 : bi;
    }
    if (nan || bi == 0x7fffffff) {
      finish(-1, -1, SAMSPEC_ST_BADROW);
      return;
    }
    if (j < S.nb && P.draft[(size_t)b * P.K + j] == bi) {
      post(kStats, j + 1, 0, NC);
      return;
    }
    finish(j, bi, 0);
    return;
  }

  if (S.kind == kStats) {
    // --- temperature softmax statistics of row j ([P3] SGLang 的实现) ---
    float lm = -__int_as_float(0x7f800000), gm = lm;
    for (int c = lane; c < NC; c += 32)
      for (int w = 0; w < kCW; ++w) {
        lm = fmaxf(lm, sm.rec[si][c][w].x);
        if (DT >= 0) gm = fmaxf(gm, sm.rec[si][c][w].z);
      }
    lm = warp_max(lm);
    if (DT >= 0) gm = warp_max(gm);
    double zt = 0.0, zg = 0.0;
    double cm_lane[2] = {0.0, 0.0};
    for (int c = lane, q = 0; c < NC; c += 32, ++q) {
      double mass = 0.0, gmass = 0.0;
      for (int w = 0; w < kCW; ++w) {
        const float4 r = sm.rec[si][c][w];
        if (r.y != 0.f) mass += (double)r.y * (double)exp2f((r.x - lm) * P.cT);
        if (r.y != r.y) mass += (double)r.y;  // keep NaN visible
        if (DT >= 0) {
          if (r.w != 0.f) gmass += (double)r.w * (double)exp2f((r.z - gm) * P.cT);
          if (r.w != r.w) gmass += (double)r.w;
        }
      }
      sm.cmass[si][c] = mass;
      if (q < 2) cm_lane[q] = mass;
      zt += mass;
      zg += gmass;
    }
    zt = warp_sum_d(zt);
    if (DT >= 0) zg = warp_sum_d(zg);
    const size_t ro = (size_t)b * (P.K + 1) + j;
    const bool bad_t = !(lm > NEG_INF) || isinf(lm) || !isfinite(zt) || !(zt > 0.0);
    const bool bad_g = DT >= 0 && j < S.nb && (!(gm > NEG_INF) || isinf(gm) || !isfinite(zg) || !(zg > 0.0));
    if (lane == 0) {
      if (P.dbg.row_m) P.dbg.row_m[ro] = lm / P.T;
      if (P.dbg.row_z) P.dbg.row_z[ro] = (float)zt;
    }
    if (bad_t || bad_g) {
      finish(-1, -1, SAMSPEC_ST_BADROW);
      return;
    }
    double pd = 0.0, ed = 0.0, qd = 1.0;
    int32_t d = -1;
    if (j < S.nb) {
      d = P.draft[(size_t)b * P.K + j];
      const float ld = load_logit(P.target, C::ST, ((size_t)b * (P.K + 1) + j) * P.V + d);
      ed = exp(((double)ld - (double)lm) / P.Td);
      pd = ed / zt;
      if (DT >= 0) {
        const float gd = load_logit(P.draftl, C::SD, ((size_t)b * P.K + j) * P.V + d);
        qd = exp(((double)gd - (double)gm) / P.Td) / zg;
      }
      float ua, ur;
      verify_coins(P.seed, P.step, (uint32_t)b, (uint32_t)j, &ua, &ur);
      if (lane == 0) {
        if (P.dbg.p_d) P.dbg.p_d[ro] = (float)pd;
        if (P.dbg.q_d) P.dbg.q_d[ro] = (float)qd;
      }
      // accept iff u * q(d) <= p(d)  ([P1] §1.1 eps <= alpha(x); [P2] §2.2)
      if ((double)ua * qd <= pd) {
        post(kStats, j + 1, 0, NC);
        return;
      }
    }
    // j is the final row: rejected (j < nb) or the bonus row (j == nb)
    float ua, ur;
    verify_coins(P.seed, P.step, (uint32_t)b, (uint32_t)j, &ua, &ur);
    if (lane == 0) {
      S.L = j;
      S.lmax = lm;
      S.gmax = gm;
      S.invZ = (float)(1.0 / zt);
      S.invZg = DT >= 0 ? (float)(1.0 / zg) : 0.f;
      S.zrow = zt;
    }
    __syncwarp();
    if (DT >= 0 && j < S.nb) {
      // residual max(0, p - q) needs both rows' full statistics: one more pass
      if (lane == 0) S.smode = 1;
      post(kResid, j, 0, NC);
      return;
    }
    // one-hot rejection: r = p with the rejected token removed; bonus: r = p.
    // Units: exp(x - m) (the row's Z is their total).
    int excl = -1;
    double sum_r = zt;
    if (j < S.nb) {
      excl = d;
      const int cd = d / C::E_TILE;
      sum_r = zt - ed;
      if (sum_r > 0.0) {
        if ((cd & 31) == lane) {
          const double nm = cm_lane[cd >> 5] - ed;
          cm_lane[cd >> 5] = nm > 0.0 ? nm : 0.0;
        }
      } else {
        excl = -1;  // residual of zero mass: fall back to p
        sum_r = zt;
      }
    }
    const double t = (double)ur * sum_r;
    // first tile whose running mass exceeds t
    double base = 0.0;
    int cstar = -1;
    double tloc = 0.0;
    for (int q = 0; q * 32 < NC && q < 2; ++q) {
      const double mine = cm_lane[q];
      const double incl = warp_incl_scan_d(mine, lane) + base;
      const unsigned hit = __ballot_sync(kFullMask, (q * 32 + lane) < NC && incl > t);
      if (hit) {
        const int src = __ffs(hit) - 1;
        cstar = q * 32 + src;
        tloc = t - (__shfl_sync(kFullMask, incl, src) - __shfl_sync(kFullMask, mine, src));
        break;
      }
      base = __shfl_sync(kFullMask, incl, 31);
    }
    if (cstar < 0) {  // rounding left the total at or below t: last tile with mass
      int lastc = -1;
      for (int q = 0; q * 32 < NC && q < 2; ++q) {
        const unsigned pos = __ballot_sync(kFullMask, (q * 32 + lane) < NC && cm_lane[q] > 0.0);
        if (pos) lastc = q * 32 + 31 - __clz(pos);
      }
      cstar = lastc < 0 ? 0 : lastc;
      const double mc = __shfl_sync(kFullMask, cm_lane[cstar >> 5], cstar & 31);
      tloc = mc;  // past the end: the scan falls back to the last positive entry
    }
    if (lane == 0) {
      S.excl = excl;
      S.smode = 0;
      S.t_local = tloc;
      S.sum_r = sum_r;
      if (P.dbg.res_mass) P.dbg.res_mass[b] = (float)(sum_r / zt);
    }
    post(kSearch, j, cstar, cstar + 1);
    return;
  }

  if (S.kind == kResid) {
    // residual mass per tile (units of p) from the second pass over row L
    double cm_lane[2] = {0.0, 0.0};
    double tot = 0.0;
    for (int c = lane, q = 0; c < NC; c += 32, ++q) {
      double m = 0.0;
      for (int w = 0; w < kCW; ++w) m += (double)sm.rec[si][c][w].x;
      if (q < 2) cm_lane[q] = m;
      tot += m;
    }
    tot = warp_sum_d(tot);
    float ua, ur;
    verify_coins(P.seed, P.step, (uint32_t)b, (uint32_t)S.L, &ua, &ur);
    int smode = 1;
    double sum_r = tot;
    if (!(tot > 0.0) || !isfinite(tot)) {
      // zero residual: sample p itself from the statistics pass's tile masses
      smode = 0;
      sum_r = S.zrow;
      for (int c = lane, q = 0; c < NC && q < 2; c += 32, ++q) cm_lane[q] = sm.cmass[si][c];
    }
    const double t = (double)ur * sum_r;
    double base = 0.0;
    int cstar = -1;
    double tloc = 0.0;
    for (int q = 0; q * 32 < NC && q < 2; ++q) {
      const double mine = cm_lane[q];
      const double incl = warp_incl_scan_d(mine, lane) + base;
      const unsigned hit = __ballot_sync(kFullMask, (q * 32 + lane) < NC && incl > t);
      if (hit) {
        const int src = __ffs(hit) - 1;
        cstar = q * 32 + src;
        tloc = t - (__shfl_sync(kFullMask, incl, src) - __shfl_sync(kFullMask, mine, src));
        break;
      }
      base = __shfl_sync(kFullMask, incl, 31);
    }
    if (cstar < 0) {
      int lastc = -1;
      for (int q = 0; q * 32 < NC && q < 2; ++q) {
        const unsigned pos = __ballot_sync(kFullMask, (q * 32 + lane) < NC && cm_lane[q] > 0.0);
        if (pos) lastc = q * 32 + 31 - __clz(pos);
      }
      cstar = lastc < 0 ? 0 : lastc;
      tloc = __shfl_sync(kFullMask, cm_lane[cstar >> 5], cstar & 31);
    }
    if (lane == 0) {
      S.smode = smode;
      S.excl = -1;
      S.t_local = tloc;
      S.sum_r = sum_r;
      if (P.dbg.res_mass) P.dbg.res_mass[b] = (float)(smode ? sum_r : 1.0);
    }
    post(kSearch, S.L, cstar, cstar + 1);
    return;
  }

  if (S.kind == kSearch) {
    // --- CDF scan inside the chosen tile, ascending token id ---
    const int stg = S.search_stage;
    const Tag tg = sm.tag[stg];
    const unsigned char* stage = stages + (size_t)stg * kStageBytes;
    const double t = S.t_local;
    const float rw = lane < kCW ? sm.rec[si][0][lane].x : 0.f;
    const double incl = warp_incl_scan_d((double)rw, lane);
    unsigned hit = __ballot_sync(kFullMask, lane < kCW && incl > t);
    int ws;
    double tw;
    if (hit) {
      ws = __ffs(hit) - 1;
      tw = t - (__shfl_sync(kFullMask, incl, ws) - __shfl_sync(kFullMask, (double)rw, ws));
    } else {
      const unsigned pos = __ballot_sync(kFullMask, lane < kCW && rw > 0.f);
      ws = pos ? 31 - __clz(pos) : 0;
      tw = 1e300;  // past the end of the slice: take its last positive entry
    }
    Slice<TT, DT> sl;
    load_slice<TT, DT>(sl, P, stage, tg, ws, lane);
    // per-vector sums in index order: vector i of lane l covers slice elements
    // (i * 32 + l) * VEC .. + VEC - 1
    int token = -1;
    double tt = tw;
    int last_pos = -1;
#pragma unroll
    for (int i = 0; i < C::VPL; ++i) {
      const int e = ws * C::SL + (i * 32 + lane) * C::VEC;
      float r[C::VEC];
      double s_l = 0.0;
#pragma unroll
      for (int k = 0; k < C::VEC; ++k) {
        r[k] = (e + k < tg.nel) ? resid_elem<TT, DT>(sl, i, k, tg.elem0 + e + k, S, P.cT) : 0.f;
        s_l += (double)r[k];
        if (r[k] > 0.f) last_pos = tg.elem0 + e + k;
      }
      const double li = warp_incl_scan_d(s_l, lane);
      const double row_total = __shfl_sync(kFullMask, li, 31);
      if (token < 0 && row_total > tt) {
        const unsigned h2 = __ballot_sync(kFullMask, li > tt);
        const int ls = __ffs(h2) - 1;
        double tl = tt - (__shfl_sync(kFullMask, li, ls) - __shfl_sync(kFullMask, s_l, ls));
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
          if (found >= 0) found = tg.elem0 + e + found;
        }
        found = __shfl_sync(kFullMask, found, ls);
        if (found >= 0) token = found;
      }
      if (token < 0) tt -= row_total;
    }
    if (token < 0) {  // fell off the end: last positive entry of the slice / tile
      int lp = last_pos;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) lp = max(lp, __shfl_xor_sync(kFullMask, lp, o));
      token = lp >= 0 ? lp : tg.elem0 + ws * C::SL;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive_cnt(&sm.empty[stg], kCW);  // release the held stage
    finish(S.L, token, 0);
    return;
  }
}

template <int TT, int DT, bool GREEDY>
__global__ void __launch_bounds__(kThreads, 1) verify_kernel(const VParams P) {
  using C = Cfg<TT, DT>;
  extern __shared__ __align__(1024) unsigned char dsm[];
  Smem& sm = *reinterpret_cast<Smem*>(dsm);
  unsigned char* stages = dsm + ((sizeof(Smem) + 1023) & ~(size_t)1023);
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
    sm.prod_done = 0;
    sm.abort = 0;
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
      load_slice<TT, DT>(sl, P, stage, tg, warp, lane);
      if (tg.kind != kSearch) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[cs]);
      }
      const bool full = tg.nel == C::E_TILE;
      float4 rec = make_float4(0.f, 0.f, 0.f, 0.f);
      if (tg.kind == kStats) {
        if (GREEDY) {
          rec = full ? reduce_greedy<TT, DT, true>(sl, warp, lane, tg.nel, tg.elem0)
                     : reduce_greedy<TT, DT, false>(sl, warp, lane, tg.nel, tg.elem0);
        } else {
          const float2 a = full ? reduce_softmax<TT, DT, true, false>(sl, warp, lane, tg.nel, P.cT)
                                : reduce_softmax<TT, DT, false, false>(sl, warp, lane, tg.nel, P.cT);
          rec.x = a.x;
          rec.y = a.y;
          if (DT >= 0 && tg.has_draft) {
            const float2 g = full ? reduce_softmax<TT, DT, true, true>(sl, warp, lane, tg.nel, P.cT)
                                  : reduce_softmax<TT, DT, false, true>(sl, warp, lane, tg.nel, P.cT);
            rec.z = g.x;
            rec.w = g.y;
          }
        }
      } else if (tg.kind == kResid) {
        rec.x = full ? reduce_resid<TT, DT, true>(sl, warp, lane, tg.nel, S, P.cT)
                     : reduce_resid<TT, DT, false>(sl, warp, lane, tg.nel, S, P.cT);
      } else {  // kSearch
        rec.x = full ? reduce_search<TT, DT, true>(sl, warp, lane, tg.nel, tg.elem0, S, P.cT)
                     : reduce_search<TT, DT, false>(sl, warp, lane, tg.nel, tg.elem0, S, P.cT);
      }
      if (lane == 0) {
        sm.rec[tg.slot][tg.chunk - S.c0][warp] = rec;
        __threadfence_block();
        const int total = (S.c1 - S.c0) * kCW;
        const int old = atomicAdd(&S.cnt, 1);
        if (old == total - 1) {
          S.cnt = 0;
          if (tg.kind == kSearch) S.search_stage = cs;
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
      bool more = true;
      uint64_t t_idle = gtimer();
      for (;;) {
        if (vload(&sm.abort)) break;
        int si = -1;
        for (int s = 0; s < kSlots && si < 0; ++s)
          if (vload(&sm.slot[s].state) == kReady) si = s;
        if (si < 0 && more) {
          for (int s = 0; s < kSlots && si < 0; ++s) {
            if (vload(&sm.slot[s].state) != kEmpty) continue;
            const uint32_t b = atomicAdd(&P.ws[0], 1u);
            if (b >= (uint32_t)P.B) {
              more = false;
              break;
            }
            Slot& S = sm.slot[s];
            int nb = P.draft_len ? P.draft_len[b] : P.K;
            bool bad = nb < 0 || nb > P.K;
            for (int jj = 0; !bad && jj < nb; ++jj) {
              const int32_t d = P.draft[(size_t)b * P.K + jj];
              bad = d < 0 || d >= P.V;
            }
            S.b = (int32_t)b;
            S.nb = bad ? 0 : nb;
            S.j = 0;
            S.L = 0;
            S.cnt = 0;
            if (bad) {
              S.kind = kInvalid;
              __threadfence_block();
              vstore(&S.state, kDone);
              continue;  // look for another empty slot
            }
            S.kind = kStats;
            S.c0 = 0;
            S.c1 = P.NC;
            si = s;
          }
        }
        if (si < 0) {
          bool all_empty = true;
          for (int s = 0; s < kSlots; ++s) all_empty &= vload(&sm.slot[s].state) == kEmpty;
          if (!more && all_empty) break;
          if (gtimer() - t_idle > kWaitNs) {
            vstore(&sm.abort, 1);
            break;
          }
          __nanosleep(64);
          continue;
        }
        __threadfence_block();
        Slot& S = sm.slot[si];
        vstore(&S.state, kIssued);
        const int kind = S.kind, b = S.b, j = S.j;
        // the draft model's row is needed for rows with a draft (j < n_b):
        // statistics, the residual pass, and a residual search
        const bool with_draft =
            DT >= 0 && j < S.nb && (kind != kSearch || S.smode == 1);
        bool ok = true;
        for (int c = S.c0; c < S.c1 && ok; ++c) {
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
            uint32_t bytes = bt;
            const uint32_t bd = with_draft ? (uint32_t)nel * C::SD : 0u;
            bytes += bd;
            mbar_arrive_expect_tx(&sm.full[ps], bytes);
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
        // sequences nobody will finish: report them
        for (uint32_t b = atomicAdd(&P.ws[0], 1u); b < (uint32_t)P.B; b = atomicAdd(&P.ws[0], 1u))
          write_result(P, (int)b, -1, -1, SAMSPEC_ST_TIMEOUT);
      }
      __threadfence_block();
      vstore(&sm.prod_done, 1);
    }
  } else if (warp == kCtrlWarp) {
    // -------------------------------- control -------------------------------
    uint64_t t_idle = gtimer();
    for (;;) {
      int si = -1;
      if (lane == 0) {
        for (int s = 0; s < kSlots && si < 0; ++s)
          if (vload(&sm.slot[s].state) == kDone) si = s;
      }
      si = __shfl_sync(kFullMask, si, 0);
      if (si >= 0) {
        __threadfence_block();
        control_handle<TT, DT, GREEDY>(P, sm, stages, si, lane);
        t_idle = gtimer();
        continue;
      }
      int stop = 0;
      if (lane == 0) {
        if (vload(&sm.abort)) {
          stop = 1;
        } else if (vload(&sm.prod_done)) {
          bool all_empty = true;
          for (int s = 0; s < kSlots; ++s) all_empty &= vload(&sm.slot[s].state) == kEmpty;
          stop = all_empty;
        } else if (gtimer() - t_idle > kWaitNs) {
          vstore(&sm.abort, 1);
          stop = 1;
        }
      }
      stop = __shfl_sync(kFullMask, stop, 0);
      if (stop) break;
      __nanosleep(64);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (sm.abort) {
      // sequences still held by this CTA's slots
      for (int s = 0; s < kSlots; ++s)
        if (sm.slot[s].state != kEmpty) write_result(P, sm.slot[s].b, -1, -1, SAMSPEC_ST_TIMEOUT);
    }
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
  const size_t head = (sizeof(Smem) + 1023) & ~(size_t)1023;
  // Device properties and the kernel's shared-memory opt-in are set up once per
  // device, so that later launches make no runtime calls besides the launch
  // itself (safe inside stream capture).
  constexpr int kMaxDev = 64;
  static int max_smem[kMaxDev] = {0}, sms[kMaxDev] = {0};
  static bool attr_done[kMaxDev] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return SAMSPEC_ECUDA;
  if (sms[dev] == 0) {
    if (cudaDeviceGetAttribute(&max_smem[dev], cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return SAMSPEC_ECUDA;
  }
  int ns = (int)((max_smem[dev] - (int)head) / kStageBytes);
  if (ns > kMaxStages) ns = kMaxStages;
  if (ns < 2) return SAMSPEC_ESIZE;
  P.NS = ns;
  const size_t smem = head + (size_t)ns * kStageBytes;
  auto kern = verify_kernel<TT, DT, GREEDY>;
  if (!attr_done[dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return SAMSPEC_ECUDA;
    attr_done[dev] = true;
  }
  const int grid = P.B < sms[dev] ? P.B : sms[dev];
  kern<<<grid, kThreads, smem, stream>>>(P);
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
  return cudaMemsetAsync(d_workspace, 0, 256, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
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
  return greedy ? dispatch<true>(P, target_dtype, ddt, s) : dispatch<false>(P, target_dtype, ddt, s);
}

int spec_uniforms(int32_t B, int32_t K, uint64_t seed, uint64_t step, float* d_u,
                  samspec_stream_t stream) {
  if (!d_u || B < 1 || K < 0 || K > 32) return SAMSPEC_EINVAL;
  const int64_t n = (int64_t)B * (K + 1);
  uniforms_kernel<<<(unsigned)((n + 255) / 256), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      B, K, seed, step, d_u);
  return cudaGetLastError() == cudaSuccess ? SAMSPEC_OK : SAMSPEC_ECUDA;
}

}  // extern "C"
