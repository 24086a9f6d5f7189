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
//   warp 24 (producer) issues 1-D bulk copies (cp.async.bulk, the TMA engine)
//       of 48 KB vocab tiles of the rows its sequence slots ask for into a
//       ring of shared-memory stages, completion counted on mbarriers;
//   warps 0-23 (consumers) each take a 1/24 slice ("warp slice") of every
//       tile into registers, release the stage, and reduce the slice to a
//       record -- its max, an integer exponent reference R and the sum of
//       2^(l log2(e)/T - R), or (greedy) its max -- then count the tile done;
//   warps 25-27 (control, one per sequence slot) claim sequences from a
//       global counter and merge each tile's 24 records as soon as they land
//       (running max, reference and compensated float-pair mass, and the mass
//       before each tile), so the row's statistics are ready when its last
//       tile is; they draw the Philox coins, decide accept/reject and post the
//       next row.  After the final row a control warp resamples: the tile
//       prefix masses and slice records locate the warp slice holding
//       u' * sum(r), and only that 3-6 KB slice is read again (from L2) and
//       scanned in ascending token order.
// Three slots keep the producer streaming while control warps decide.  Tiles
// of 48 KB (4 ring stages) measured faster than 24-32 KB tiles: the per-tile
// work of producer, consumers and control is amortised over more logits.
// 24 consumer warps measured faster than 8, 12 or 16: a warp's per-tile chain
// (load, max, exponentials, warp reductions, record) is latency-bound, and
// more warps overlap more chains.  The producer writes per-tile fields the
// consumers would otherwise recompute per slice (record index, full and
// non-empty slices, the warp holding the draft token or a tree's children),
// and the first tiles of a CTA's first sequence are requested at launch.
// Small batches run as thread-block clusters whose CTAs stream a sequence's
// tiles round robin; with fp32 targets or draft logits the tile's last
// consumer warp merges the records there, so one control warp does not set
// the pace.  Launches use programmatic dependent launch.  Every wait is
// bounded by a global-timer deadline; a CTA that runs out of time marks its
// sequences SAMSPEC_ST_TIMEOUT, lets its copies in flight land and exits.

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>

#include "common.cuh"
#include "philox.cuh"
#include "sampling.cuh"
#include "samspec.h"

namespace samspec {
namespace {

constexpr int kCW = 24;              // consumer warps
constexpr int kProdWarp = kCW;       // producer warp
constexpr int kCtrlWarp = kCW + 1;   // first control warp (one per slot)
constexpr int kSlots = 3;
constexpr int kThreads = (kCW + 1 + kSlots) * 32;
constexpr int kStageBytes = 49152;
constexpr int kMaxStages = 6;
constexpr int kMinStages = 3;
constexpr int kMaxChunks = 48;
constexpr int kMaxChunksDraft = 32;  // with draft logits: both arrays' records must fit
constexpr uint64_t kWaitNs = 2000000000ull;   // 2 s per pipeline wait (default)
constexpr uint64_t kDrainNs = 2000000000ull;  // 2 s for copies in flight to land after an abort
constexpr uint32_t kSuspendNs = 20000;  // longest suspension of one producer wait on a stage
// the pipeline waits' limit for launches made from now on (test hook)
std::atomic<uint64_t> g_wait_ns{kWaitNs};
constexpr size_t kVerifyWorkspaceBytes = 256;  // work counters: claims, exits, error bits

// kSkip: a tile requested ahead for a job that did not come (its stage is
// released unread)
enum Kind : int32_t { kStats = 0, kResid = 1, kSkip = 2, kExit = 3 };
enum State : int32_t { kEmpty = 0, kReady = 1, kIssued = 2 };

struct VParams {
  const unsigned char* target;
  const unsigned char* draftl;
  const int32_t* draft;
  const int32_t* draft_len;
  int32_t B, K, V;
  float T, cT;  // cT = log2(e) / T, rounded to fp32
  float cTl;    // cT + cTl = log2(e) / T to about 2^-48 relative
  double Td, cTd;
  uint64_t seed, step;
  int32_t* accept_len;
  int32_t* out_token;
  int32_t* emit;
  int32_t* emit_len;
  int32_t* status;
  spec_verify_debug dbg;
  uint32_t* ws;  // [0] claim counter, [1] CTA exit counter, [2] error bits
  int32_t NC, NS;
  int32_t G;         // CTAs per thread-block cluster: a sequence's tiles are shared among them
  uint64_t wait_ns;  // limit of every pipeline wait
  int32_t direct;  // 1: plain loads instead of bulk copies (unaligned rows)
  // draft trees (K = N - 1, row n scores the token after node n's path)
  const int32_t* ttok;  // [B, N] node tokens (node 0: the verified context)
  const int32_t* tfc;   // [B, N] first child, -1: none
  const int32_t* tns;   // [B, N] next sibling, -1: none
  int32_t* path;        // [B, N] accepted node indices, -1 after
  // per-request sampling parameters: temperature [B] and the cut of each row
  // [B, K+1] (logits below it are left out; -inf: none; NaN: bad parameters)
  const float* seqT;
  const float* tau;
};

struct __align__(16) Tag {
  // the consumers' words first: job kind; record index of (slot, tile, warp
  // 0); warp slices wholly inside the tile, and with any element of it
  int32_t kind, rbase, nfull, nany;
  // the warp whose slice holds the row's draft token (statistics pass of a
  // drafted row; -1: none in this tile) and the token's index in the tile
  int32_t dwarp, dtile, slot, chunk;
  int32_t nel, elem0, has_draft, b;
  int32_t j, dtok;  // the row's draft token (statistics pass of a drafted row), else -1
  uint32_t cwarps;  // trees: the warps whose slices hold one of the node's children
  int32_t pad;
};

struct Slot {
  int32_t state;  // State, accessed with volatile loads/stores
  int32_t kind;   // kind of the current job (kStats: row j; kResid: row L)
  int32_t b, j, nb, L;
  int32_t smode;  // residual pass: 1 -> max(0, p - q) in units of p;
                  //                0 -> p in units of exp(x - m)
  float lmax, gmax, invZ, invZg;
  int32_t dtok;   // draft token of the current row (-1 for the bonus row)
  float xd, gd;   // target / draft logit at dtok, captured by the consumers
  int32_t age;    // claim order inside the CTA: the producer serves the oldest first
  // draft trees: depth of the current row, its children's tokens (sibling
  // order; left out of the sums like a linear draft) and their logits
  int32_t depth, nex;
  int32_t ex[32];
  float cx[32];
  // per-request sampling: the sequence's temperature, log2(e)/T as cT + cTl,
  // and the cut of the row in flight
  float T, cT, cTl, tau;
};

// One warp-slice record: softmax statistics of the target (a) and draft (b)
// rows; greedy {max, 0, NaN seen, 0} in a; residual pass {rh, rl, 0, 0} in a.
// In shared memory the a parts of all slots, tiles and slices come first, then
// (with draft logits only) the b parts in the same order.
struct Rec {
  float4 a, b;
};
template <int DT>
__host__ __device__ constexpr size_t rec_bytes_of(int NC) {
  return (size_t)(DT >= 0 ? 2 : 1) * kSlots * NC * kCW * sizeof(float4);
}

struct Smem {
  Slot slot[kSlots];
  Tag tag[kMaxStages];
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  int32_t stage_parity[kMaxStages];  // parity of the last issue per stage
  int32_t abort;
  int32_t prod_idle;    // the producer has issued every posted job
  int32_t jobs_issued;  // jobs whose tiles the producer has all issued
  int32_t ctrl_exited;  // control warps that have finished
  int32_t claims;       // sequences claimed by this CTA
  int32_t pool_left;    // sequences not yet claimed, as of this CTA's last claim
  int32_t claim_lock;   // one control warp claims at a time
  int32_t pool_done;    // a claim found no sequence left: idle slots leave
  int32_t claims_ended; // this CTA has counted itself out of the claim counter
  uint64_t tile_bar[kSlots][kMaxChunks];  // one phase per job: the kCW records of a tile
  float4 pre[kSlots][kMaxChunks][2];     // control: mass before each tile {hi, lo, ref, 0}
                                         // (clusters: first the tile's summary)
  // clusters: the tile's warps that have stored their records (the last one
  // merges them; its summary goes to the leader's `pre` entry of the tile)
  uint32_t tcnt[kSlots][kMaxChunks];
};

// Sets this CTA's abort flag, and (clusters) every other CTA's of the cluster.
__device__ __forceinline__ void set_abort(Smem& sm, int G) {
  vstore(&sm.abort, 1);
  if (G > 1) {
    const uint32_t me = cluster_rank();
    for (int r = 0; r < G; ++r)
      if ((uint32_t)r != me) st_cluster_u32(cluster_map(&sm.abort, (uint32_t)r), 1u);
  }
}

// Called once a CTA will claim no more sequences from the shared counter
// (once per CTA): counts the CTA out, and the last CTA out resets the
// counters for the next launch on this workspace.  Done as soon as the
// CTA's claiming ends, not at its exit, so the global atomics are off the
// end of the launch.
__device__ __forceinline__ void end_claims(const VParams& P, Smem& sm, int G) {
  if (gridDim.x / (uint32_t)G >= (uint32_t)P.B) return;  // the counter is not used
  if (atomicExch(&sm.claims_ended, 1) != 0) return;
  __threadfence();
  if (atomicAdd(&P.ws[1], 1u) == gridDim.x - 1) {
    P.ws[0] = 0;
    P.ws[1] = 0;
    __threadfence();
  }
}

// Words of a slot that the other CTAs of a cluster need for a job (kind ..
// depth; the state word is written after them).
constexpr int kSlotSyncWords = 15;

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

// packed fp32 pairs (Blackwell f32x2 arithmetic)
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ void upk2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// ---- compensated (double-float) sums -------------------------------------------
// A value is hi + lo with |lo| <= ulp(hi) / 2; additions carry the rounding
// error of every step (Knuth's TwoSum), so a sum of fp32 terms keeps about 44
// significant bits.
struct DF {
  float hi, lo;
};
__device__ __forceinline__ DF df_add(DF x, DF y) {
  const float s = x.hi + y.hi;
  const float bb = s - x.hi;
  const float e = (x.hi - (s - bb)) + (y.hi - bb);
  const float lo = e + (x.lo + y.lo);
  const float hi = s + lo;
  return {hi, lo - (hi - s)};
}
__device__ __forceinline__ DF df_neg(DF x) { return {-x.hi, -x.lo}; }
__device__ __forceinline__ DF df_sub(DF x, DF y) { return df_add(x, df_neg(y)); }
// x <= y for normalised pairs (|lo| at most half an ulp of hi)
__device__ __forceinline__ bool df_le(DF x, DF y) {
  return x.hi < y.hi || (x.hi == y.hi && x.lo <= y.lo);
}
// x * 2^k: one multiply by the power of two when 2^k is a normal float,
// ldexpf otherwise (exact while the result stays normal)
__device__ __forceinline__ float scale2(float x, int k) {
  if (k >= -126 && k <= 127) return x * __int_as_float((k + 127) << 23);
  return ldexpf(x, k);
}
__device__ __forceinline__ DF df_scale(DF x, int k) { return {scale2(x.hi, k), scale2(x.lo, k)}; }
// x * a with the product's rounding error carried (FMA two-product)
__device__ __forceinline__ DF df_mul_f(DF x, float a) {
  const float p = x.hi * a;
  const float e = fmaf(x.hi, a, -p) + x.lo * a;
  const float hi = p + e;
  return {hi, e - (hi - p)};
}
__device__ __forceinline__ float df_f(DF x) { return x.hi + x.lo; }
// Warp sum of lane values in [0, 2^11) as a float pair: each value splits
// into a multiple of 2^-10 (rounding by the 1.5 * 2^13 constant) and the
// remainder (|r| <= 2^-11).  The multiples sum exactly as integers (below
// 2^26); the remainders sum as integers in units of 2^-34 (each rounded by at
// most 2^-35, so the total is off by at most 2^-30).  One warp reduction
// instruction each.
__device__ __forceinline__ DF split_warp_sum(float v) {
  const float hi = (v + 12288.f) - 12288.f;
  const float r = v - hi;
  const uint32_t k1 = __reduce_add_sync(kFullMask, (uint32_t)(hi * 1024.f));
  const int32_t k2 = (int32_t)__reduce_add_sync(kFullMask, (uint32_t)__float2int_rn(r * 0x1p34f));
  const float a = __uint2float_rz(k1);               // k1 with its lowest bits cut (k1 < 2^26)
  const float ea = (float)(k1 - __float2uint_rz(a));  // the cut bits, exact
  const float ah = a * 0x1p-10f;
  const float small = fmaf(ea, 0x1p-10f, (float)k2 * 0x1p-34f);
  const float sum = ah + small;
  const float bb = sum - ah;
  return {sum, (ah - (sum - bb)) + (small - bb)};
}
// Warp sum of lane values in [0, 32] whose total is at least 1/2, as a float
// pair: each value is rounded to a multiple of 2^-26 (exact for values of at
// least 1/8, at most 2^-27 off below that), and the integers are summed
// exactly in two 16-bit halves, one warp reduction each.  The total is off by
// at most 2^-22, a relative 2^-21.
__device__ __forceinline__ DF fixed_warp_sum(float v) {
  const uint32_t k = __float2uint_rn(v * 0x1p26f);
  const uint32_t kh = __reduce_add_sync(kFullMask, k >> 16);     // < 2^20
  const uint32_t kl = __reduce_add_sync(kFullMask, k & 0xFFFFu);  // < 2^21
  const float hi = (float)kh * 0x1p-10f;  // both exact
  const float lo = (float)kl * 0x1p-26f;
  const float sum = hi + lo;  // hi > 1/4 > lo: the error of the add is exact
  return {sum, lo - (sum - hi)};
}
// NaN-propagating warp maximum in one warp reduction instruction
__device__ __forceinline__ float warp_max_nan(float v) {
  float m;
  asm("redux.sync.max.NaN.f32 %0, %1, 0xffffffff;" : "=f"(m) : "f"(v));
  return m;
}
__device__ __forceinline__ DF df_warp_sum(DF a) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const DF o2 = {__shfl_xor_sync(kFullMask, a.hi, o), __shfl_xor_sync(kFullMask, a.lo, o)};
    a = df_add(a, o2);
  }
  return a;
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
  // elements (2p, 2p + 1) as a packed fp32 pair
  __device__ __forceinline__ uint64_t pair(int p) const {
    if (ES == 4) return pk2(__uint_as_float(w[2 * p]), __uint_as_float(w[2 * p + 1]));
    return pk2(bf16_lo(w[p]), bf16_hi(w[p]));
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
  static constexpr int E_TILE = DT < 0 ? kStageBytes / ST : (ST == SD ? kStageBytes / (2 * ST) : kStageBytes / 8);
  static constexpr int SL = E_TILE / kCW;        // elements per warp slice
  static constexpr int VPL = SL / (32 * VEC);    // vectors per lane per array
  static constexpr int DOFF = E_TILE * ST;       // byte offset of the draft part
  static_assert(VPL >= 1 && VPL * 32 * VEC * kCW == E_TILE, "tile shape");
  static_assert((VEC & (VEC - 1)) == 0, "vector length is a power of two");
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
// memory for the control warp, lane-major: lane l holds the slice's elements
// [l * EPL, (l + 1) * EPL) (EPL = SL / 32), vector i covering elements
// l * EPL + i * VEC + k.  Returns the slice's element count.
template <int TT, int DT>
__device__ __forceinline__ int load_slice_lanes(Slice<TT, DT>& s, const VParams& P, int b, int L,
                                                int c, int w, bool with_draft, int lane) {
  using C = Cfg<TT, DT>;
  constexpr int EPL = C::SL / 32;
  const int s0 = c * C::E_TILE + w * C::SL;
  const size_t rt = ((size_t)b * (P.K + 1) + L) * (size_t)P.V;
  const size_t rd = ((size_t)b * P.K + L) * (size_t)P.V;
#pragma unroll
  for (int i = 0; i < C::VPL; ++i) {
    const int e = s0 + lane * EPL + i * C::VEC;  // vocab index
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
  constexpr int ES = DRAFT_ARRAY ? C::SD : C::ST;
  if constexpr (FULL && ES == 2) {
    // bf16: packed maxima over every word of the lane, one unpack at the end
    constexpr int W = C::VEC / 2;
    uint32_t a = DRAFT_ARRAY ? s.d[0].w[0] : s.t[0].w[0];
#pragma unroll
    for (int i = 0; i < C::VPL; ++i)
#pragma unroll
      for (int q = 0; q < W; ++q)
        if (i > 0 || q > 0) a = bf16x2_max_nan(a, DRAFT_ARRAY ? s.d[i].w[q] : s.t[i].w[q]);
    m = fmax_nan(bf16_lo(a), bf16_hi(a));
  } else {
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
  }
  return m;
}

// greedy record: {slice max, 0, NaN seen}.  The first position of the row's
// maximum is found afterwards, in the one warp slice that holds it.
template <int TT, int DT, bool FULL>
__device__ __forceinline__ float4 reduce_greedy(const Slice<TT, DT>& s, int w, int lane, int nel) {
  const float m = warp_max_nan(lane_max<TT, DT, FULL, false>(s, w, lane, nel));
  if (m != m) return make_float4(0.f, 0.f, 1.f, 0.f);
  return make_float4(m, 0.f, 0.f, 0.f);
}

// Sum of 2^(x * cT - R) over a lane's elements of a full slice: pairs of
// elements through packed FFMA / FADD, one MUFU ex2 each.  MASK: elements
// whose bit i * VEC + k is set in xm count zero.
template <int TT, int DT, bool DRAFT_ARRAY, bool MASK, bool THR = false>
__device__ __forceinline__ float packed_exp_sum(const Slice<TT, DT>& s, float cT, float R, uint64_t xm,
                                                float tau = 0.f) {
  using C = Cfg<TT, DT>;
  const uint64_t c2 = pk2(cT, cT), nr2 = pk2(-R, -R);
  uint64_t part[C::VPL];
#pragma unroll
  for (int i = 0; i < C::VPL; ++i) {
    uint64_t v[C::VEC / 2];
#pragma unroll
    for (int p = 0; p < C::VEC / 2; ++p) {
      const uint64_t xv = DRAFT_ARRAY ? s.d[i].pair(p) : s.t[i].pair(p);
      const uint64_t y = fma2(xv, c2, nr2);
      float y0, y1;
      upk2(y, y0, y1);
      float e0 = ex2_approx(y0), e1 = ex2_approx(y1);
      if (THR) {  // logits below the cut count zero
        float x0, x1;
        upk2(xv, x0, x1);
        if (!(x0 >= tau)) e0 = 0.f;
        if (!(x1 >= tau)) e1 = 0.f;
      }
      if (MASK) {
        if ((xm >> (i * C::VEC + 2 * p)) & 1ull) e0 = 0.f;
        if ((xm >> (i * C::VEC + 2 * p + 1)) & 1ull) e1 = 0.f;
      }
      v[p] = pk2(e0, e1);
    }
#pragma unroll
    for (int h = C::VEC / 4; h >= 1; h >>= 1)
#pragma unroll
      for (int p = 0; p < h; ++p) v[p] = add2(v[p], v[p + h]);
    part[i] = v[0];
  }
  // pairwise over the lane's VPL vectors (VPL need not be a power of two)
#pragma unroll
  for (int h = 1; h < C::VPL; h <<= 1)
#pragma unroll
    for (int i = 0; i + h < C::VPL; i += 2 * h) part[i] = add2(part[i], part[i + h]);
  float lo, hi;
  upk2(part[0], lo, hi);
  return lo + hi;
}

// Softmax record of one array of the slice: {m, R, z, 0} with m the slice
// max, R = ceil(fl(m * cT)) an integer exponent reference and z the fp32 sum
// of 2^fl(x * cT - R) over the slice (every term in (0, ~1]).
// Records of one row combine by exact power-of-two scaling 2^(R - max R), so no
// per-record exponential enters the row's masses.  The element with tile index
// `excl` (the row's draft token, added back exactly by the control warp) is
// left out; the caller passes it to the warp whose slice holds it only, and
// -1 to the others.  An all -inf slice gives {-inf, -inf, 0, 0}; NaN gives
// NaNs.
template <int TT, int DT, bool FULL, bool DRAFT_ARRAY, bool MULTI = false, bool THR = false>
__device__ __forceinline__ float4 reduce_softmax(const Slice<TT, DT>& s, int w, int lane, int nel,
                                                 float cT, int excl, uint64_t xm = 0,
                                                 float tau = 0.f, bool any_xm = true) {
  using C = Cfg<TT, DT>;
  const float NEG_INF = -__int_as_float(0x7f800000);
  const float QNAN = __int_as_float(0x7fc00000);
  const float m = warp_max_nan(lane_max<TT, DT, FULL, DRAFT_ARRAY>(s, w, lane, nel));
  if (!(m > NEG_INF))
    return m != m ? make_float4(QNAN, QNAN, QNAN, QNAN) : make_float4(NEG_INF, NEG_INF, 0.f, 0.f);
  const float R = ceilf(m * cT);
  float z;
  // `excl`: one element left out (tile index, or -1).  MULTI: xm marks the
  // lane's elements left out (bit i * VEC + k), e.g. a tree node's children;
  // the warp takes the masked path if any lane has one (any_xm false: the
  // caller knows that none has)
  const bool single = excl >= 0;
  const bool has_excl = single || (MULTI && any_xm && __any_sync(kFullMask, xm != 0));
  // THR: logits below tau (a per-request cut) are left out too
  const bool cut = THR && tau > NEG_INF;
  if (FULL && !has_excl && !cut) {
    // the slice's maximum is in the sum: its term is in (1/2, 1], so the
    // total is at least 1/2 and each lane's at most its element count
    static_assert(C::SL / 32 <= 32, "at most 32 elements per lane");
    z = packed_exp_sum<TT, DT, DRAFT_ARRAY, false>(s, cT, R, 0);
    const DF zz = fixed_warp_sum(z);
    return make_float4(m, R, zz.hi, zz.lo);
  } else if (THR && FULL && !has_excl) {
    z = packed_exp_sum<TT, DT, DRAFT_ARRAY, false, true>(s, cT, R, 0, tau);
  } else if (MULTI && FULL && !single) {
    z = packed_exp_sum<TT, DT, DRAFT_ARRAY, true>(s, cT, R, xm);
  } else {
    float part[C::VPL];
#pragma unroll
    for (int i = 0; i < C::VPL; ++i) {
      const int e = w * C::SL + (i * 32 + lane) * C::VEC;
      float v[C::VEC];
#pragma unroll
      for (int k = 0; k < C::VEC; ++k) {
        const float x = DRAFT_ARRAY ? s.d[i].at(k) : s.t[i].at(k);
        bool keep = e + k < nel && e + k != excl;
        if (MULTI) keep &= !((xm >> (i * C::VEC + k)) & 1ull);
        if (THR) keep &= x >= tau;
        v[k] = keep ? ex2_approx(fmaf(x, cT, -R)) : 0.f;
      }
#pragma unroll
      for (int h = C::VEC / 2; h >= 1; h >>= 1)
#pragma unroll
        for (int k = 0; k < h; ++k) v[k] += v[k + h];
      part[i] = v[0];
    }
#pragma unroll
    for (int h = 1; h < C::VPL; h <<= 1)
#pragma unroll
      for (int i = 0; i + h < C::VPL; i += 2 * h) part[i] += part[i + h];
    z = part[0];
  }
  // lane sums in fp32; the warp's 32 lane sums as a float pair (z, w)
  const DF zz = split_warp_sum(z);
  return make_float4(m, R, zz.hi, zz.lo);
}

// Residual weight of one element, the same expression in the residual pass and
// in the resample scan (so a slice's mass and its scan agree):
//   smode 0: 2^fl(x * cT - RL), units 2^RL;
//   smode 1: max(0, 2^fl(x * cT - RL) * invZ - 2^fl(g * cT - RG) * invZg), units of p.
template <int TT, int DT>
__device__ __forceinline__ float resid_elem(const Slice<TT, DT>& s, int i, int k, int smode,
                                            float RL, float RG, float invZ, float invZg, float cT) {
  const float pe = ex2_approx(fmaf(s.t[i].at(k), cT, -RL));
  if (smode == 0) return pe;
  float g = 0.f;
  if (DT >= 0) g = s.d[i].at(k);
  const float qe = ex2_approx(fmaf(g, cT, -RG));
  return fmaxf(0.f, pe * invZ - qe * invZg);
}

// resid_elem for one logit pair (x target, g draft).
__device__ __forceinline__ float resid_val(float x, float g, int smode, float RL, float RG,
                                           float invZ, float invZg, float cT) {
  const float pe = ex2_approx(fmaf(x, cT, -RL));
  if (smode == 0) return pe;
  const float qe = ex2_approx(fmaf(g, cT, -RG));
  return fmaxf(0.f, pe * invZ - qe * invZg);
}

// residual-pass record: sum of r over the slice as a float pair {hi, lo, 0, 0}
template <int TT, int DT, bool FULL>
__device__ __forceinline__ float4 reduce_resid(const Slice<TT, DT>& s, int w, int lane, int nel,
                                               const Slot& S, float cT) {
  using C = Cfg<TT, DT>;
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < C::VPL; ++i) {
    const int e = w * C::SL + (i * 32 + lane) * C::VEC;
    float part = 0.f;
#pragma unroll
    for (int k = 0; k < C::VEC; ++k)
      if (FULL || e + k < nel)
        part += resid_elem<TT, DT>(s, i, k, S.smode, S.lmax, S.gmax, S.invZ, S.invZg, cT);
    acc += part;
  }
  const DF a = split_warp_sum(acc);
  return make_float4(a.hi, a.lo, 0.f, 0.f);
}

// ---- outputs ---------------------------------------------------------------
__device__ void write_result(const VParams& P, int b, int L, int out, int st) {
  if (P.path)
    for (int t = 0; t <= P.K; ++t) P.path[(size_t)b * (P.K + 1) + t] = -1;
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

// First lane in [0, n) whose inclusive running sum of v exceeds t, or -1;
// *before receives the running sum ahead of that lane.  Sums are carried as
// float pairs (about 48 significant bits).
__device__ __forceinline__ int warp_find(DF v, DF t, int n, int lane, DF* before) {
  DF x = lane < n ? v : DF{0.f, 0.f};
  DF incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const DF y = {__shfl_up_sync(kFullMask, incl.hi, o), __shfl_up_sync(kFullMask, incl.lo, o)};
    if (lane >= o) incl = df_add(incl, y);
  }
  const unsigned hit = __ballot_sync(kFullMask, lane < n && !df_le(incl, t));
  if (!hit) return -1;
  const int src = __ffs(hit) - 1;
  const DF bef = df_sub(incl, x);
  *before = {__shfl_sync(kFullMask, bef.hi, src), __shfl_sync(kFullMask, bef.lo, src)};
  return src;
}

__device__ __forceinline__ float warp_incl_scan_f(float v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(kFullMask, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

// ---- control warp ------------------------------------------------------------
// Clusters: which side merges a tile's kCW records.  With fp32 targets, or a
// draft array to merge as well, tiles complete faster than one control warp
// merges them, so the tile's last consumer warp does it (records stay in the
// streaming CTA).  bf16 one-hot rows keep the control warp's merge (records
// go to the leader): there the extra work in the consumers costs more.
template <int TT, int DT, bool CL>
__host__ __device__ constexpr bool consumers_merge() {
  return CL && (TT == 0 || DT >= 0);
}

// ---- tile summaries: the warp-wide part of merging a tile's kCW records ----
// Lane w < kCW holds record w of the tile, the other lanes a neutral record.
// Softmax array: {max logit, max reference Rc, the tile's mass in units 2^Rc
// as a float pair}, the max logit NaN when a record holds a NaN (it makes the
// row bad whatever the maxima are).
__device__ __forceinline__ float4 softmax_tile_summary(float4 r) {
  const float NEG_INF = -__int_as_float(0x7f800000);
  const bool nan = __any_sync(kFullMask, r.x != r.x || r.z != r.z);
  const float mc = nan ? __int_as_float(0x7fc00000) : warp_max_nan(r.x);
  const float Rc = warp_max_nan(r.y);
  DF v = {0.f, 0.f};
  if (Rc != NEG_INF && r.z != 0.f) v = df_scale(DF{r.z, r.w}, (int)(r.y - Rc));
  const DF t = df_warp_sum(v);
  return make_float4(mc, Rc, t.hi, t.lo);
}
// Greedy: {tile max M, first slice holding M, 1 if a record saw a NaN, 0}.
__device__ __forceinline__ float4 greedy_tile_summary(float4 r, int lane) {
  const float NEG_INF = -__int_as_float(0x7f800000);
  const float m = lane < kCW ? r.x : NEG_INF;
  const bool nan = __any_sync(kFullMask, lane < kCW && r.z != 0.f);
  const float M = warp_max_nan(m);
  const unsigned h = __ballot_sync(kFullMask, lane < kCW && m == M);
  return make_float4(M, (float)(h ? __ffs(h) - 1 : 0), nan ? 1.f : 0.f, 0.f);
}
// Residual pass: the tile's residual mass as a float pair {hi, lo, 0, 0}.
__device__ __forceinline__ float4 resid_tile_summary(float4 r, int lane) {
  const DF t = df_warp_sum(lane < kCW ? DF{r.x, r.y} : DF{0.f, 0.f});
  return make_float4(t.hi, t.lo, 0.f, 0.f);
}

// Records of a slot are indexed r = c * kCW + w (tile c, warp slice w); a
// merge of tile c gives lane w < kCW the record (c, w).

// 2^(x * log2(e)/T - R) for one token (R an integer-valued reference),
// accurate to a few fp32 ulp: log2(e)/T is carried as cT + cTl, x * cT and
// its rounding error exactly (FMA), the difference to R by TwoSum, and the
// integer part of the exponent split off before exp2f.
__device__ __forceinline__ float exp_ref(float x, float R, float cT, float cTl) {
  const float yh = x * cT;
  const float e1 = fmaf(x, cT, -yh) + x * cTl;
  const float s = yh - R;
  const float bb = s - yh;
  const float e2 = (yh - (s - bb)) + (-R - bb);
  const float si = rintf(s);
  return ldexpf(exp2f((s - si) + (e1 + e2)), (int)fmaxf(si, -300.f));
}

template <int TT, int DT, bool GREEDY, bool TREE = false, bool SAMP = false, bool CL = false>
struct Control {
  using C = Cfg<TT, DT>;
  static constexpr int EPL = C::SL / 32;  // slice elements per lane (lane-major loads)
  const VParams& P;
  Smem& sm;
  const float4* rec;  // a parts [kSlots][NC][kCW], then (draft logits) b parts
  int lane, si;
  bool more;
  int32_t tok;        // lane t holds draft token t of the slot's sequence
                      // (trees: the token of node t)
  int32_t par_;       // trees: parent of node `lane`
  int32_t pathv;      // trees: the node accepted at depth `lane`
  float ua, ur;       // coins of the row in flight (drawn while it streams)
  bool first_;        // slot 0's first claim: sequence blockIdx.x, no atomic

  __device__ Control(const VParams& p, Smem& s, const float4* r, int l, int slot)
      : P(p), sm(s), rec(r), lane(l), si(slot), more(true), tok(-1), par_(-1), pathv(-1),
        ua(0.f), ur(0.f), first_(slot == 0) {
    reset_row();
  }

  // temperature terms and the row's cut: per sequence with sampling
  // parameters, else the launch's
  __device__ float cT_() const { return SAMP ? sm.slot[si].cT : P.cT; }
  __device__ float cTl_() const { return SAMP ? sm.slot[si].cTl : P.cTl; }
  __device__ float T_() const { return SAMP ? sm.slot[si].T : P.T; }
  __device__ double cTd_() const {
    return SAMP ? (double)sm.slot[si].cT + (double)sm.slot[si].cTl : P.cTd;
  }
  __device__ float tau_() const { return SAMP ? sm.slot[si].tau : -__int_as_float(0x7f800000); }

  // Record (tile c, slice w) of the slot.  When the consumers merge, it
  // lives in the shared memory of the CTA that streamed tile c (rank c mod G).
  __device__ Rec R(int c, int w) const {
    const size_t i = ((size_t)si * P.NC + c) * kCW + w;
    const size_t ib = (size_t)kSlots * P.NC * kCW + i;
    Rec r;
    const uint32_t owner = consumers_merge<TT, DT, CL>() ? (uint32_t)(c % P.G) : 0u;
    if (owner != 0) {
      r.a = ld_cluster_f32x4(cluster_map(&rec[i], owner));
      r.b = DT >= 0 ? ld_cluster_f32x4(cluster_map(&rec[ib], owner)) : make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
      r.a = rec[i];
      r.b = DT >= 0 ? rec[ib] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    return r;
  }

  // Outputs of sequence b, written by the warp's lanes in parallel (lane t
  // holds draft token t).
  __device__ void finish(int b, int L, int out, int st) {
    if (TREE) {
      // the accepted path's nodes, then their tokens and the final token
      const int32_t pt = __shfl_sync(kFullMask, tok, pathv & 31);
      if (lane <= P.K) {
        if (P.path) P.path[(size_t)b * (P.K + 1) + lane] = (!st && lane < L) ? pathv : -1;
        if (P.emit)
          P.emit[(size_t)b * (P.K + 1) + lane] = st ? -1 : (lane < L ? pt : (lane == L ? out : -1));
      }
    } else if (P.emit) {
      int32_t* e = P.emit + (size_t)b * (P.K + 1);
      if (lane <= P.K) e[lane] = st ? -1 : (lane < L ? tok : (lane == L ? out : -1));
      if (P.K == 32 && lane == 0) e[32] = st ? -1 : (L == 32 ? out : -1);
    }
    if (lane == 0) {
      P.accept_len[b] = st ? -1 : L;
      P.out_token[b] = st ? -1 : out;
      if (P.status) P.status[b] = st;
      if (P.emit_len) P.emit_len[b] = st ? 0 : L + 1;
    }
    __syncwarp();
  }

  __device__ void release() {
    if (lane == 0) vstore(&sm.slot[si].state, kEmpty);
    __syncwarp();
  }

  // Clusters: the job's words of the slot go to the same slot of every other
  // CTA of the cluster (their producers stream the job's other tiles and
  // their consumers read the residual pass's terms), then its ready state.
  __device__ void publish() {
    const int32_t* w = reinterpret_cast<const int32_t*>(&sm.slot[si]);
    const int G = CL ? P.G : 1;
    for (int k = lane; k < (G - 1) * kSlotSyncWords; k += 32) {
      const int r = 1 + k / kSlotSyncWords, q = 1 + k % kSlotSyncWords;
      st_cluster_u32(cluster_map(w + q, (uint32_t)r), (uint32_t)w[q]);
    }
    fence_cluster();
    __syncwarp();
    if (lane >= 1 && lane < G) st_cluster_u32(cluster_map(&sm.slot[si].state, (uint32_t)lane), (uint32_t)kReady);
    __syncwarp();
  }

  // Posts row j for the producer, then draws the row's coins while it streams.
  __device__ void post(int kind, int j) {
    Slot& S = sm.slot[si];
    if (TREE) {
      // row j is node j; its children (sibling order = index order) are the
      // candidates, left out of the row's sums
      const unsigned cm = __ballot_sync(kFullMask, lane <= P.K && par_ == j && lane > 0);
      if ((cm >> lane) & 1u) S.ex[__popc(cm & ((1u << lane) - 1u))] = tok;
      __syncwarp();  // the lanes' entries before lane 0 publishes the job
      if (lane == 0) {
        S.kind = kind;
        S.j = j;
        S.dtok = -1;
        S.nex = kind == kStats ? __popc(cm) : 0;
        __threadfence_block();
        vstore(&S.state, kReady);
      }
      __syncwarp();
      if (!GREEDY) verify_coins(P.seed, P.step, (uint32_t)S.b, (uint32_t)S.depth, &ua, &ur);
      return;
    }
    const int32_t dt = __shfl_sync(kFullMask, tok, j & 31);
    if (lane == 0) {
      S.kind = kind;
      S.j = j;
      S.dtok = (kind == kStats && j < S.nb) ? dt : -1;
      if (SAMP) S.tau = P.tau[(size_t)S.b * (P.K + 1) + j];
      __threadfence_block();
    }
    __syncwarp();
    if (CL) publish();
    if (lane == 0) vstore(&S.state, kReady);
    __syncwarp();
    if (!GREEDY) verify_coins(P.seed, P.step, (uint32_t)S.b, (uint32_t)j, &ua, &ur);
  }

  // Trees: node `lane` of sequence b into registers (token, parent), and the
  // shape checks: every link points to a larger index below N, every node
  // n >= 1 is linked exactly once, node 0 has no sibling, tokens lie in
  // [0, V), siblings carry distinct tokens.
  __device__ bool tree_load(int b) {
    const int N = P.K + 1;
    const bool in = lane < N;
    const size_t o = (size_t)b * N + lane;
    tok = in && lane > 0 ? P.ttok[o] : -1;
    const int32_t fc = in ? P.tfc[o] : -1;
    const int32_t ns = in ? P.tns[o] : -1;
    bool bad = in && ((lane > 0 && (tok < 0 || tok >= P.V)) || (fc != -1 && (fc <= lane || fc >= N)) ||
                      (ns != -1 && (ns <= lane || ns >= N)) || (lane == 0 && ns != -1));
    if (__any_sync(kFullMask, bad)) return false;
    // parents, in index order: node c is the first child of some n, or the
    // next sibling of some s < c (whose parent is already known)
    par_ = -1;
    for (int c = 1; c < N; ++c) {
      const unsigned f = __ballot_sync(kFullMask, in && fc == c);
      const unsigned g = __ballot_sync(kFullMask, in && ns == c);
      if (__popc(f) + __popc(g) != 1) return false;
      const int32_t pc = f ? (__ffs(f) - 1) : __shfl_sync(kFullMask, par_, __ffs(g) - 1);
      if (lane == c) par_ = pc;
    }
    // distinct tokens among siblings
    const unsigned long long key = in && lane > 0
                                       ? ((unsigned long long)(uint32_t)par_ << 32) | (uint32_t)tok
                                       : (0xFFFFFFFFull << 32) | (uint32_t)lane;
    const unsigned same = __match_any_sync(kFullMask, key);
    return !__any_sync(kFullMask, in && lane > 0 && __popc(same) > 1);
  }

  // Claims sequences until one with valid drafts lands in the slot (or none
  // are left: the slot stays empty).
  __device__ void refill() {
    Slot& S = sm.slot[si];
    while (more) {
      uint32_t b = 0;
      if (lane == 0) {
        // cluster x's first sequence is x (clusters <= B); later ones come
        // from the shared counter, past the first `ncl` (none when the
        // clusters cover the batch: the counter is then never touched)
        const uint32_t G = CL ? (uint32_t)P.G : 1u;
        const uint32_t ncl = gridDim.x / G;
        // (claims are made under the CTA's claim lock: once one found the
        // pool empty, none is made again)
        b = first_ ? blockIdx.x / G
                   : (ncl >= (uint32_t)P.B || vload(&sm.pool_done)) ? (uint32_t)P.B
                                                                     : ncl + atomicAdd(&P.ws[0], 1u);
        vstore(&sm.pool_left, b >= (uint32_t)P.B ? 0 : P.B - 1 - (int)b);
        // no sequence left: none beyond this one either when the clusters
        // cover the batch, so the slots leave without another claim
        if (b >= (uint32_t)P.B || ncl >= (uint32_t)P.B) vstore(&sm.pool_done, 1);
        if (b >= (uint32_t)P.B) end_claims(P, sm, (int)G);
      }
      first_ = false;
      b = __shfl_sync(kFullMask, b, 0);
      if (b >= (uint32_t)P.B) {
        more = false;
        break;
      }
      if (TREE) {
        if (!tree_load((int)b)) {
          finish((int)b, -1, -1, SAMSPEC_ST_BADDRAFT);
          continue;
        }
        pathv = -1;
        if (lane == 0) {
          S.b = (int32_t)b;
          S.nb = 0;
          S.L = 0;
          S.depth = 0;
          S.age = atomicAdd(&sm.claims, 1);
        }
        __syncwarp();
        post(kStats, 0);
        return;
      }
      const int nb = P.draft_len ? P.draft_len[b] : P.K;
      tok = (lane < P.K) ? P.draft[(size_t)b * P.K + lane] : -1;
      bool bad = nb < 0 || nb > P.K || (lane < nb && (tok < 0 || tok >= P.V));
      if (__any_sync(kFullMask, bad)) {
        finish((int)b, -1, -1, SAMSPEC_ST_BADDRAFT);
        continue;
      }
      if (SAMP) {
        // the sequence's temperature, and every row's cut: a temperature not
        // > 0 and finite, or a NaN cut (top_p not > 0), refuses the sequence
        const float Tb = P.seqT[b];
        const float tj = lane <= P.K ? P.tau[(size_t)b * (P.K + 1) + lane] : 0.f;
        const bool nan_cut = __any_sync(kFullMask, tj != tj);
        if (nan_cut || !(Tb > 0.f) || !(Tb < __int_as_float(0x7f800000))) {
          finish((int)b, -1, -1, SAMSPEC_ST_BADPARAM);
          continue;
        }
        if (lane == 0) {
          const double cTd = 1.4426950408889634 / (double)Tb;
          S.T = Tb;
          S.cT = (float)cTd;
          S.cTl = (float)(cTd - (double)S.cT);
        }
      }
      if (lane == 0) {
        S.b = (int32_t)b;
        S.nb = nb;
        S.L = 0;
        S.age = atomicAdd(&sm.claims, 1);
      }
      __syncwarp();
      post(kStats, 0);
      return;
    }
  }

  // ---- running row state, updated tile by tile while the row streams -------
  // Softmax arrays (f = 0 target, 1 draft): max logit, exponent reference
  // (max slice reference so far) and the compensated mass of the tiles merged
  // so far in units of 2^ref; the mass before each tile goes to sm.pre.
  struct Run {
    float mx, ref;
    DF sum;
    bool nan;
  };
  Run run[2];
  // greedy: row max, and the first slice holding it (tile * kCW + slice)
  float gmax_;
  int gfirst_;
  bool gnan_;

  __device__ void reset_row() {
    const float NEG_INF = -__int_as_float(0x7f800000);
#pragma unroll
    for (int f = 0; f < 2; ++f) run[f] = Run{NEG_INF, NEG_INF, DF{0.f, 0.f}, false};
    gmax_ = NEG_INF;
    gfirst_ = -1;
    gnan_ = false;
  }

  // Adds tile c's slices of array f (records in lanes 0..15) to run[f].
  // The summary of array f of tile c: computed here from the records, or,
  // in clusters, the one the tile's last warp wrote into pre[si][c][f] (read
  // by every lane before lane 0 overwrites that entry).
  __device__ float4 summary(int c, int f) {
    if (consumers_merge<TT, DT, CL>()) {
      const float4 v = sm.pre[si][c][f];
      __syncwarp();
      return v;
    }
    const float NEG_INF = -__int_as_float(0x7f800000);
    const Rec r = R(c, lane < kCW ? lane : 0);
    const float4 x = lane < kCW ? (f ? r.b : r.a) : make_float4(NEG_INF, NEG_INF, 0.f, 0.f);
    if (GREEDY) return greedy_tile_summary(x, lane);
    if (sm.slot[si].kind != kStats) return resid_tile_summary(x, lane);
    return softmax_tile_summary(x);
  }

  __device__ void merge_softmax(int c, int f) {
    const float NEG_INF = -__int_as_float(0x7f800000);
    const float4 sv = summary(c, f);
    const bool nan = sv.x != sv.x;
    const float mc = sv.x, Rc = sv.y;
    const DF t = {sv.z, sv.w};  // the tile's mass over its slices, units 2^Rc
    Run& R_ = run[f];
    if (lane == 0) sm.pre[si][c][f] = make_float4(R_.sum.hi, R_.sum.lo, R_.ref, 0.f);
    R_.nan |= nan;
    R_.mx = fmaxf(R_.mx, mc);
    // the reference follows every finite tile reference, with or without mass
    // (a row whose only token left in the sums is the draft itself keeps a
    // finite reference for the draft's exponential)
    if (Rc != NEG_INF && Rc > R_.ref) {  // a larger reference: rescale what was summed so far
      if (R_.ref != NEG_INF) {
        const int sc = (int)(R_.ref - Rc);
        R_.sum = df_scale(R_.sum, sc);
      }
      R_.ref = Rc;
    }
    if (Rc != NEG_INF && (t.hi != 0.f || t.lo != 0.f)) {
      const int sc = (int)(Rc - R_.ref);
      R_.sum = df_add(R_.sum, df_scale(t, sc));
    }
  }

  __device__ void merge_tile(int c) {
    Slot& S = sm.slot[si];
    if (c == 0) reset_row();
    if (GREEDY) {
      const float4 sv = summary(c, 0);
      gnan_ |= sv.z != 0.f;
      if (sv.x > gmax_) {  // tiles arrive in token order: keep the first maximum
        gmax_ = sv.x;
        gfirst_ = c * kCW + (int)sv.y;
      }
    } else if (S.kind == kStats) {
      merge_softmax(c, 0);
      if (DT >= 0 && S.j < S.nb) merge_softmax(c, 1);
    } else {  // residual pass: plain running sum in units of p
      const float4 sv = summary(c, 0);
      const DF t = {sv.x, sv.y};
      if (lane == 0) sm.pre[si][c][0] = make_float4(run[0].sum.hi, run[0].sum.lo, 0.f, 0.f);
      run[0].sum = df_add(run[0].sum, t);
      run[0].ref = 0.f;
    }
    __syncwarp();
  }

  // First position of value M in warp slice (c, w) of row j (greedy argmax).
  __device__ int first_index_of(int b, int j, int c, int w, float M) {
    Slice<TT, DT> sl;
    const int n = load_slice_lanes<TT, DT>(sl, P, b, j, c, w, false, lane);
    const int s0 = c * C::E_TILE + w * C::SL;
    int idx = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < C::VPL; ++i) {
      const int e = lane * EPL + i * C::VEC;
#pragma unroll
      for (int k = 0; k < C::VEC; ++k)
        if (e + k < n && sl.t[i].at(k) == M && idx == 0x7fffffff) idx = s0 + e + k;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) idx = min(idx, __shfl_xor_sync(kFullMask, idx, o));
    return idx;
  }

  // Resample scan of warp slice (c, w) of row L: the first token whose running
  // residual exceeds t (in the slice's own units: the expression its record
  // summed, resid_val, with token `excl` left out), ascending token order.
  // Each lane sums its own contiguous elements; a warp scan finds the lane;
  // that lane's elements go one per lane and a second warp scan finds the
  // token.
  __device__ int slice_scan(int b, int L, int c, int w, float t, int smode, int excl, float RL,
                            float RG, float invZ, float invZg, const int32_t* exl = nullptr,
                            int nex = 0) {
    static_assert(EPL <= 64, "one mask bit per element of a lane");
    Slice<TT, DT> sl;
    const bool with_draft = DT >= 0 && smode == 1;
    const int n = load_slice_lanes<TT, DT>(sl, P, b, L, c, w, with_draft, lane);
    const int s0 = c * C::E_TILE + w * C::SL;
    // the tokens left out of the residual (`excl` and the listed ids), as bits
    // of the lane holding them (lane-major: lane l holds l * EPL .. + EPL - 1)
    uint64_t xl = 0;
    for (int q = -1; q < nex; ++q) {
      const int o = (q < 0 ? excl : exl[q]) - s0;
      if (o >= 0 && o < n && o / EPL == lane) xl |= 1ull << (o % EPL);
    }
    float tot = 0.f;
    int last_pos = -1;
#pragma unroll
    for (int i = 0; i < C::VPL; ++i)
#pragma unroll
      for (int k = 0; k < C::VEC; ++k) {
        const int e = lane * EPL + i * C::VEC + k;
        float r = 0.f;
        if (e < n && !((xl >> (i * C::VEC + k)) & 1ull))
          r = resid_val(sl.t[i].at(k), DT >= 0 ? sl.d[i].at(k) : 0.f, smode, RL, RG, invZ, invZg, cT_());
        if (SAMP && !(sl.t[i].at(k) >= tau_())) r = 0.f;
        tot += r;
        if (r > 0.f) last_pos = s0 + e;
      }
    const float incl = warp_incl_scan_f(tot, lane);
    const unsigned hit = __ballot_sync(kFullMask, incl > t);
    if (!hit) {  // rounding put t past the slice: its last positive entry
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
        last_pos = max(last_pos, __shfl_xor_sync(kFullMask, last_pos, o));
      return last_pos >= 0 ? last_pos : s0;
    }
    const int ls = __ffs(hit) - 1;
    const uint64_t xls = __shfl_sync(kFullMask, xl, ls);
    float tl = t - __shfl_sync(kFullMask, incl - tot, ls);
    // lane ls's elements, 32 at a time in ascending order: element q to lane
    // q % 32 of round q / 32
    constexpr int kRounds = (EPL + 31) / 32;
#pragma unroll
    for (int rd = 0; rd < kRounds; ++rd) {
      float xe = 0.f, ge = 0.f;
#pragma unroll
      for (int i = 0; i < C::VPL; ++i)
#pragma unroll
        for (int k = 0; k < C::VEC; ++k) {
          const int q = i * C::VEC + k;
          if (q / 32 != rd) continue;
          const float xv = __shfl_sync(kFullMask, sl.t[i].at(k), ls);
          float gv = 0.f;
          if (DT >= 0 && with_draft) gv = __shfl_sync(kFullMask, sl.d[i].at(k), ls);
          if (lane == q % 32) {
            xe = xv;
            ge = gv;
          }
        }
      const int q = rd * 32 + lane;
      const int e = ls * EPL + q;
      float re = 0.f;
      if (q < EPL && e < n && !((xls >> q) & 1ull))
        re = resid_val(xe, ge, smode, RL, RG, invZ, invZg, cT_());
      if (SAMP && !(xe >= tau_())) re = 0.f;
      const float inc2 = warp_incl_scan_f(re, lane);
      const unsigned h2 = __ballot_sync(kFullMask, q < EPL && inc2 > tl);
      if (h2) return s0 + ls * EPL + rd * 32 + __ffs(h2) - 1;
      tl -= __shfl_sync(kFullMask, inc2, 31);
    }
    // rounding: the lane's last positive entry
    return __shfl_sync(kFullMask, last_pos, ls);
  }

  // The tile holding t: the last tile whose prefix mass (sm.pre, rescaled to
  // units of 2^ref_units) is <= t; then the warp slice from the tile's slice
  // masses (slice_mass(c, w) -> float pair, units 2^ref_units); then scan(c, w, t_w)
  // inside it.
  template <typename SliceMass, typename Scan>
  __device__ int resample(DF t, float ref_units, SliceMass slice_mass, Scan scan) {
    const int NC = P.NC;
    const float NEG_INF = -__int_as_float(0x7f800000);
    int cstar = 0;
    DF before = {0.f, 0.f};
#pragma unroll
    for (int q = 1; q >= 0; --q) {
      const int c = q * 32 + lane;
      DF bc = {0.f, 0.f};
      bool ok = false;
      if (c < NC) {
        const float4 pr = sm.pre[si][c][0];
        if (pr.z != NEG_INF && (pr.x != 0.f || pr.y != 0.f))
          bc = df_scale(DF{pr.x, pr.y}, (int)(pr.z - ref_units));
        ok = df_le(bc, t);
      }
      const unsigned h = __ballot_sync(kFullMask, ok);
      if (h) {
        const int src = 31 - __clz(h);
        cstar = q * 32 + src;
        before = {__shfl_sync(kFullMask, bc.hi, src), __shfl_sync(kFullMask, bc.lo, src)};
        break;
      }
    }
    const DF tc = df_sub(t, before);
    const DF sm_w = lane < kCW ? slice_mass(cstar, lane) : DF{0.f, 0.f};
    DF bw = {0.f, 0.f};
    int wstar = warp_find(sm_w, tc, kCW, lane, &bw);
    DF tw;
    if (wstar < 0) {  // rounding put t past the tile: its last slice with mass
      const unsigned pos = __ballot_sync(kFullMask, lane < kCW && sm_w.hi > 0.f);
      wstar = pos ? 31 - __clz(pos) : 0;
      tw = {__int_as_float(0x7f800000), 0.f};
    } else {
      tw = df_sub(tc, bw);
    }
    return scan(cstar, wstar, tw);
  }

  // Trees: node `node` accepted at the current depth; post its row.
  __device__ void advance(int node) {
    Slot& S = sm.slot[si];
    const int depth = S.depth;
    if (lane == depth) pathv = node;
    __syncwarp();
    if (lane == 0) S.depth = depth + 1;
    __syncwarp();
    post(kStats, node);
  }

  // Trees, T > 0: row j (node j) is complete.  Its children k_1 .. k_m were
  // left out of the sums; p(k_i) from their captured logits; one coin u for
  // this depth takes the first child with u <= p(k_1) + ... + p(k_i).  If
  // none, or a leaf, the final token is drawn from the row without the
  // children (the sums already leave them out).
  __device__ void tree_step(int b, int j, size_t ro) {
    Slot& S = sm.slot[si];
    const float NEG_INF = -__int_as_float(0x7f800000);
    const int nex = S.nex;
    const float lm = run[0].nan ? __int_as_float(0x7fc00000) : run[0].mx;
    const float LM = run[0].ref;
    const DF zx = run[0].sum;
    const float ek = lane < nex ? exp_ref(S.cx[lane], LM, cT_(), cTl_()) : 0.f;
    const DF ztd = df_add(zx, df_warp_sum(DF{ek, 0.f}));
    const float zt = df_f(ztd);
    const bool bad = !(lm > NEG_INF) || isinf(lm) || !isfinite(zt) || !(zt > 0.f);
    if (lane == 0) {
      if (P.dbg.row_m) P.dbg.row_m[ro] = lm / T_();
      if (P.dbg.row_z)
        P.dbg.row_z[ro] = (float)(((double)ztd.hi + (double)ztd.lo) * exp2((double)LM - (double)lm * cTd_()));
    }
    if (bad) {
      finish(b, -1, -1, SAMSPEC_ST_BADROW);
      release();
      return;
    }
    // running sum of the children's probabilities, in sibling order
    float inc = ek;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(kFullMask, inc, o);
      if (lane >= o) inc += y;
    }
    const unsigned hit = __ballot_sync(kFullMask, lane < nex && ua * zt <= inc);
    if (hit) {
      const int k = __ffs(hit) - 1;
      // the k-th child in sibling order
      const unsigned cm = __ballot_sync(kFullMask, lane <= P.K && lane > 0 && par_ == j);
      const bool mine = ((cm >> lane) & 1u) && __popc(cm & ((1u << lane) - 1u)) == k;
      advance(__ffs(__ballot_sync(kFullMask, mine)) - 1);
      return;
    }
    const int depth = S.depth;
    if (!(df_f(zx) > 0.f)) {
      // only the children carry mass (rounding): the child holding u' of it
      const unsigned h2 = __ballot_sync(kFullMask, lane < nex && ur * zt <= inc);
      const int k = h2 ? __ffs(h2) - 1 : nex - 1;
      finish(b, depth, S.ex[k], 0);
      release();
      return;
    }
    if (lane == 0 && P.dbg.res_mass) P.dbg.res_mass[b] = df_f(zx) / zt;
    const DF tt = df_mul_f(zx, ur);
    auto slice_mass = [&](int c, int w) -> DF {
      const float4 r = R(c, w).a;
      if (r.y == NEG_INF || r.z == 0.f) return DF{0.f, 0.f};
      return df_scale(DF{r.z, r.w}, (int)(r.y - LM));
    };
    auto scan = [&](int c, int w, DF tw) -> int {
      const float Rw = R(c, w).a.y;
      return slice_scan(b, j, c, w, df_f(df_scale(tw, (int)(LM - Rw))), 0, -1, Rw, 0.f, 0.f, 0.f,
                        S.ex, nex);
    };
    const int out = resample(tt, LM, slice_mass, scan);
    finish(b, depth, out, 0);
    release();
  }

  __device__ void handle() {
    Slot& S = sm.slot[si];
    const int b = S.b, j = S.j, nb = S.nb;
    const size_t ro = (size_t)b * (P.K + 1) + j;
    const float NEG_INF = -__int_as_float(0x7f800000);

    if (GREEDY) {
      const float M = gmax_;
      int idx = 0x7fffffff;
      if (!gnan_ && M != NEG_INF && gfirst_ >= 0)
        idx = first_index_of(b, j, gfirst_ / kCW, gfirst_ % kCW, M);
      const bool bad = gnan_ || idx == 0x7fffffff;
      if (lane == 0) {
        if (P.dbg.row_m) P.dbg.row_m[ro] = M;
        if (P.dbg.row_arg) P.dbg.row_arg[ro] = bad ? -1 : idx;
      }
      if (bad) {
        finish(b, -1, -1, SAMSPEC_ST_BADROW);
        release();
        return;
      }
      if (TREE) {  // follow the child holding the argmax, if there is one
        const unsigned cm = __ballot_sync(kFullMask, lane <= P.K && lane > 0 && par_ == j && tok == idx);
        if (cm) {
          advance(__ffs(cm) - 1);
          return;
        }
        finish(b, S.depth, idx, 0);
        release();
        return;
      }
      const int32_t dj = __shfl_sync(kFullMask, tok, j & 31);
      if (j < nb && dj == idx) {
        post(kStats, j + 1);
        return;
      }
      finish(b, j, idx, 0);
      release();
      return;
    }

    if (TREE && S.kind == kStats) {
      tree_step(b, j, ro);
      return;
    }

    if (S.kind == kStats) {
      // --- temperature-softmax statistics of row j from the running state:
      // row max lm, reference LM, every tile's mass scaled exactly to 2^LM ---
      const int32_t d = j < nb ? S.dtok : -1;
      const float lm = run[0].nan ? __int_as_float(0x7fc00000) : run[0].mx;
      const float LM = run[0].ref;
      const DF zx = run[0].sum;
      float gm = NEG_INF, GM = NEG_INF, egd = 0.f;
      DF zg = {0.f, 0.f};
      if (DT >= 0 && j < nb) {
        gm = run[1].nan ? __int_as_float(0x7fc00000) : run[1].mx;
        GM = run[1].ref;
        zg = run[1].sum;
        egd = exp_ref(S.gd, GM, cT_(), cTl_());  // draft model's d, units 2^GM
      }
      // one-hot: the sums leave d out (zx), so that a rejection's residual is
      // exact; with draft logits they hold every token
      // (a draft below the row's cut has probability 0)
      const float ed = (d >= 0 && (!SAMP || S.xd >= S.tau)) ? exp_ref(S.xd, LM, cT_(), cTl_()) : 0.f;
      const DF ztd = DT < 0 ? df_add(zx, DF{ed, 0.f}) : zx;
      const float zt = df_f(ztd), zgf = df_f(zg);
      const bool bad_t = !(lm > NEG_INF) || isinf(lm) || !isfinite(zt) || !(zt > 0.f);
      const bool bad_g = DT >= 0 && j < nb &&
                         (!(gm > NEG_INF) || isinf(gm) || !isfinite(zgf) || !(zgf > 0.f));
      if (lane == 0) {
        if (P.dbg.row_m) P.dbg.row_m[ro] = lm / T_();
        // Z relative to the row max: sum exp(x/T - m) = zt * 2^(LM - lm log2(e)/T)
        if (P.dbg.row_z)
          P.dbg.row_z[ro] = (float)(((double)ztd.hi + (double)ztd.lo) * exp2((double)LM - (double)lm * cTd_()));
      }
      if (bad_t || bad_g) {
        finish(b, -1, -1, SAMSPEC_ST_BADROW);
        release();
        return;
      }
      if (j < nb) {
        const float pd = ed / zt;
        const float qd = DT >= 0 ? egd / zgf : 1.f;
        if (lane == 0) {
          if (P.dbg.p_d) P.dbg.p_d[ro] = pd;
          if (P.dbg.q_d) P.dbg.q_d[ro] = qd;
        }
        // accept iff u * q(d) <= p(d)  (eps <= alpha(x) with alpha = min(1, p/q))
        if (ua * qd <= pd) {
          post(kStats, j + 1);
          return;
        }
      }
      // j is the final row L: rejected (j < nb) or the bonus row (j == nb)
      if (DT >= 0 && j < nb) {
        // residual max(0, p - q) needs both rows' full statistics: one more pass
        if (lane == 0) {
          S.L = j;
          S.lmax = LM;
          S.gmax = GM;
          S.invZ = 1.f / zt;
          S.invZg = 1.f / zgf;
          S.smode = 1;
        }
        __syncwarp();
        post(kResid, j);
        return;
      }
      // one-hot rejection: r = p without the rejected token, which the slice
      // sums already leave out; bonus row (no draft): r = p.  Units 2^LM.
      if (j < nb && !(df_f(zx) > 0.f)) {
        // every other token has zero mass: p is concentrated on d itself
        if (lane == 0 && P.dbg.res_mass) P.dbg.res_mass[b] = 1.f;
        finish(b, j, d, 0);
        release();
        return;
      }
      if (lane == 0 && P.dbg.res_mass) P.dbg.res_mass[b] = df_f(zx) / zt;
      const DF tt = df_mul_f(zx, ur);
      auto slice_mass = [&](int c, int w) -> DF {
        const float4 r = R(c, w).a;
        if (r.y == NEG_INF || r.z == 0.f) return DF{0.f, 0.f};
        return df_scale(DF{r.z, r.w}, (int)(r.y - LM));
      };
      auto scan = [&](int c, int w, DF tw) -> int {
        // the slice's own units: 2^R_w
        const float Rw = R(c, w).a.y;
        return slice_scan(b, j, c, w, df_f(df_scale(tw, (int)(LM - Rw))), 0, d, Rw, 0.f, 0.f, 0.f);
      };
      const int out = resample(tt, LM, slice_mass, scan);
      finish(b, j, out, 0);
      release();
      return;
    }

    // kResid: the running residual mass of row L and its tile prefixes
    const int L = S.L;
    const float tot = df_f(run[0].sum);
    if (S.smode == 1 && (!(tot > 0.f) || !isfinite(tot))) {
      // zero residual (impossible in exact arithmetic): sample p instead
      if (lane == 0) S.smode = 0;
      __syncwarp();
      post(kResid, L);
      return;
    }
    if (lane == 0 && P.dbg.res_mass) P.dbg.res_mass[b] = S.smode ? tot : 1.f;
    const DF tt = df_mul_f(run[0].sum, ur);
    auto slice_mass = [&](int c, int w) -> DF { return DF{R(c, w).a.x, R(c, w).a.y}; };
    auto scan = [&](int c, int w, DF tw) -> int {
      return slice_scan(b, L, c, w, df_f(tw), S.smode, -1, S.lmax, S.gmax, S.invZ, S.invZg);
    };
    const int out = resample(tt, 0.f, slice_mass, scan);
    finish(b, L, out, 0);
    release();
  }
};

// CL: launched in thread-block clusters of P.G CTAs that share each
// sequence's tiles (small batches); without it, one CTA per sequence and no
// cluster code at all in the instantiation.
template <int TT, int DT, bool GREEDY, bool TREE = false, bool SAMP = false, bool CL = false>
__global__ void __launch_bounds__(kThreads, 1) verify_kernel(const VParams P) {
  using C = Cfg<TT, DT>;
  extern __shared__ __align__(1024) unsigned char dsm[];
  Smem& sm = *reinterpret_cast<Smem*>(dsm);
  const size_t rec_off = (sizeof(Smem) + 15) & ~(size_t)15;
  float4* rec = reinterpret_cast<float4*>(dsm + rec_off);
  const size_t rec_bytes = rec_bytes_of<DT>(P.NC);
  unsigned char* stages = dsm + ((rec_off + rec_bytes + 1023) & ~(size_t)1023);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int NS = P.NS;
  const int G = CL ? P.G : 1;                 // CTAs of this cluster (1: no cluster)
  const uint32_t crank = CL ? cluster_rank() : 0u;  // 0: the leader, whose control warps decide

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kCW);
      sm.stage_parity[s] = -1;
    }
    for (int s = 0; s < kSlots; ++s) {
      sm.slot[s].state = kEmpty;
    }
    sm.abort = 0;
    sm.prod_idle = 0;
    sm.jobs_issued = 0;
    sm.ctrl_exited = 0;
    sm.claims = 0;
    sm.pool_left = P.B;
    sm.claim_lock = 0;
    sm.pool_done = 0;
    sm.claims_ended = 0;
    mbar_fence_init();
  }
  // tile barriers: each consumer warp arrives once per tile of a job
  // (other CTAs of a cluster arrive on them: each init is fenced at cluster scope)
  if (threadIdx.x < kSlots * kMaxChunks) {
    // one arrival when the tile's last consumer warp merges its records
    mbar_init(&sm.tile_bar[threadIdx.x / kMaxChunks][threadIdx.x % kMaxChunks],
              consumers_merge<TT, DT, CL>() ? 1 : kCW);
    sm.tcnt[threadIdx.x / kMaxChunks][threadIdx.x % kMaxChunks] = 0;
    mbar_fence_init();
  }
  __syncthreads();
  // clusters: no CTA writes into another's shared memory before it is set up
  if (G > 1) cluster_sync_all();
  // programmatic dependent launch: the next kernel on the stream may start
  // its own set-up now; this one touches global memory only once the
  // kernel before it has completed and its writes are visible
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");

  if (warp < kCW) {
    // ------------------------------ consumers ------------------------------
    int cs = 0;
    uint32_t cph = 0;
    bool nxt_ready = false;  // the next stage was seen full before this slice's record
    for (;;) {
      bool ok = true;
      if (!nxt_ready && !mbar_try_wait(&sm.full[cs], cph)) {
        const uint64_t t0 = gtimer();
        while (!mbar_try_wait(&sm.full[cs], cph)) {
          if (vload(&sm.abort) || gtimer() - t0 > P.wait_ns) {
            ok = false;
            break;
          }
        }
      }
      if (!ok) {
        if (lane == 0) set_abort(sm, G);
        break;
      }
      const Tag tg = sm.tag[cs];
      if (tg.kind == kExit) break;
      if (tg.kind == kSkip) {
        nxt_ready = false;
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[cs]);
        if (++cs == NS) {
          cs = 0;
          cph ^= 1;
        }
        continue;
      }
      Slot& S = sm.slot[tg.slot];
      const unsigned char* stage = stages + (size_t)cs * kStageBytes;
      // a row's last tile is partial: slices past its end hold nothing (their
      // records are empty), slices wholly inside it take the unmasked path
      const bool none = warp >= tg.nany;
      const bool full = warp < tg.nfull;
      Slice<TT, DT> sl;
      if (!none) load_slice_tile<TT, DT>(sl, P, stage, tg, warp, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[cs]);
      Rec r;
      r.a = make_float4(0.f, 0.f, 0.f, 0.f);
      r.b = r.a;
      if (none) {
        // the records of an all -inf slice; a residual slice holds no mass
        const float NEG_INF = -__int_as_float(0x7f800000);
        if (tg.kind == kStats) {
          r.a = make_float4(NEG_INF, GREEDY ? 0.f : NEG_INF, 0.f, 0.f);
          r.b = make_float4(NEG_INF, NEG_INF, 0.f, 0.f);
        }
      } else if (tg.kind == kStats) {
        if (GREEDY) {
          r.a = full ? reduce_greedy<TT, DT, true>(sl, warp, lane, tg.nel)
                     : reduce_greedy<TT, DT, false>(sl, warp, lane, tg.nel);
        } else {
          // one-hot drafts: the row's draft token is left out of the sums
          // (tile index, or -1), so the residual of a rejection is exact
          const int ex = (DT < 0 && warp == tg.dwarp) ? tg.dtile : -1;
          if (TREE) {
            // a tree node's children are left out of the sums: the lane
            // holding one keeps its logit and marks it in its mask
            static_assert(C::VPL * C::VEC <= 64, "one mask bit per element of a lane");
            // (only the warps whose slices hold a child look them up)
            const bool holds = (tg.cwarps >> warp) & 1u;
            const int nex = holds ? S.nex : 0;
            uint64_t xm = 0;
            for (int k = 0; k < nex; ++k) {
              const int o = S.ex[k] - tg.elem0 - warp * C::SL;
              if (o >= 0 && o < C::SL && o + warp * C::SL < tg.nel) {
                const int v = o / C::VEC, kk = o % C::VEC;
                if ((v & 31) == lane) {
                  const int ii = v >> 5;
                  float x = 0.f;
#pragma unroll
                  for (int i = 0; i < C::VPL; ++i)
#pragma unroll
                    for (int q = 0; q < C::VEC; ++q)
                      if (i == ii && q == kk) x = sl.t[i].at(q);
                  S.cx[k] = x;
                  xm |= 1ull << (ii * C::VEC + kk);
                }
              }
            }
            r.a = full ? reduce_softmax<TT, DT, true, false, true>(sl, warp, lane, tg.nel, P.cT, -1, xm, 0.f, holds)
                       : reduce_softmax<TT, DT, false, false, true>(sl, warp, lane, tg.nel, P.cT, -1, xm, 0.f, holds);
          } else {
          if (SAMP) {  // the sequence's temperature; logits below the row's cut left out
            const float cTs = S.cT, th = S.tau;
            r.a = full ? reduce_softmax<TT, DT, true, false, false, true>(sl, warp, lane, tg.nel, cTs, ex, 0, th)
                       : reduce_softmax<TT, DT, false, false, false, true>(sl, warp, lane, tg.nel, cTs, ex, 0, th);
          } else {
            r.a = full ? reduce_softmax<TT, DT, true, false>(sl, warp, lane, tg.nel, P.cT, ex)
                       : reduce_softmax<TT, DT, false, false>(sl, warp, lane, tg.nel, P.cT, ex);
          }
          }
          if (DT >= 0 && tg.has_draft) {
            r.b = full ? reduce_softmax<TT, DT, true, true>(sl, warp, lane, tg.nel, P.cT, ex)
                       : reduce_softmax<TT, DT, false, true>(sl, warp, lane, tg.nel, P.cT, ex);
          }
        }
      } else {  // kResid
        r.a = full ? reduce_resid<TT, DT, true>(sl, warp, lane, tg.nel, S, P.cT)
                   : reduce_resid<TT, DT, false>(sl, warp, lane, tg.nel, S, P.cT);
      }
      if (warp == tg.dwarp) {
        // the lane holding the draft token keeps its logits for the decision
        const int o = tg.dtile - warp * C::SL;
        const int v = o / C::VEC, kk = o % C::VEC;
        if ((v & 31) == lane) {
          const int ii = v >> 5;
          float x = 0.f, g = 0.f;
#pragma unroll
          for (int i = 0; i < C::VPL; ++i)
#pragma unroll
            for (int k = 0; k < C::VEC; ++k)
              if (i == ii && k == kk) {
                x = sl.t[i].at(k);
                if (DT >= 0 && tg.has_draft) g = sl.d[i].at(k);
              }
          if (G == 1) {
            S.xd = x;
            S.gd = g;
          } else {  // the leader's slot takes the decision
            st_cluster_u32(cluster_map(&S.xd, 0), __float_as_uint(x));
            st_cluster_u32(cluster_map(&S.gd, 0), __float_as_uint(g));
            fence_cluster();
          }
        }
      }
      if (!CL) {
        // streaming batches: test the next stage now, so that the loop's
        // next wait costs nothing when its tile has landed (small batches,
        // whose next tile is rarely there yet, skip the extra test)
        const int ncs = cs + 1 == NS ? 0 : cs + 1;
        nxt_ready = mbar_test_wait(&sm.full[ncs], cs + 1 == NS ? cph ^ 1u : cph);
      }
      __syncwarp();
      int last = 0;
      if (lane == 0) {
        const int ri = tg.rbase + warp;
        // release: the record (and the captured logits) before the arrival
        if (G == 1) {
          rec[ri] = r.a;
          if (DT >= 0) rec[(size_t)kSlots * P.NC * kCW + ri] = r.b;
          mbar_arrive(&sm.tile_bar[tg.slot][tg.chunk]);
        } else if (consumers_merge<TT, DT, CL>()) {
          // the tile's last warp (all of them are this CTA's) merges
          rec[ri] = r.a;
          if (DT >= 0) rec[(size_t)kSlots * P.NC * kCW + ri] = r.b;
          __threadfence_block();
          last = atomicAdd(&sm.tcnt[tg.slot][tg.chunk], 1u) == (uint32_t)kCW - 1u;
        } else {  // into the cluster leader's records, on its tile barrier
          st_cluster_f32x4(cluster_map(&rec[ri], 0), r.a);
          if (DT >= 0) st_cluster_f32x4(cluster_map(&rec[(size_t)kSlots * P.NC * kCW + ri], 0), r.b);
          mbar_arrive_cluster(cluster_map(&sm.tile_bar[tg.slot][tg.chunk], 0));
        }
      }
      if (consumers_merge<TT, DT, CL>() && __shfl_sync(kFullMask, last, 0)) {
        // Clusters: the last of the tile's warps reduces its kCW records (all
        // in this CTA's shared memory) to the tile's summary, for the leader's
        // control warp, which then only folds it into the row's running state.
        __threadfence_block();
        __syncwarp();
        const float NEG_INF = -__int_as_float(0x7f800000);
        const size_t base = ((size_t)tg.slot * P.NC + tg.chunk) * kCW;
        const bool two = DT >= 0 && tg.kind == kStats && tg.has_draft;
        float4 ra = make_float4(NEG_INF, NEG_INF, 0.f, 0.f), rb = ra;
        if (lane < kCW) {
          ra = rec[base + lane];
          if (two) rb = rec[(size_t)kSlots * P.NC * kCW + base + lane];
        }
        float4 s0, s1 = make_float4(0.f, 0.f, 0.f, 0.f);
        if (GREEDY) {
          s0 = greedy_tile_summary(ra, lane);
        } else if (tg.kind == kStats) {
          s0 = softmax_tile_summary(ra);
          if (two) s1 = softmax_tile_summary(rb);
        } else {
          s0 = resid_tile_summary(ra, lane);
        }
        if (lane == 0) {
          st_cluster_f32x4(cluster_map(&sm.pre[tg.slot][tg.chunk][0], 0), s0);
          if (two) st_cluster_f32x4(cluster_map(&sm.pre[tg.slot][tg.chunk][1], 0), s1);
          // the counter for the slot's next job (posted only after the control
          // warp has seen this arrival)
          sm.tcnt[tg.slot][tg.chunk] = 0;
          mbar_arrive_cluster(cluster_map(&sm.tile_bar[tg.slot][tg.chunk], 0));
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
      // Row 0 of the CTA's first sequence is read whatever its drafts are (it
      // scores draft 0, or it is the bonus row), so its first tiles are
      // requested at once, before the control warp has claimed the sequence
      // and loaded its drafts.  Their stages are published (tag, then the
      // producer's arrival) when the job is posted; if another job comes
      // first (the sequence's drafts were bad), they are released unread.
      int npre = 0;
      bool early = false;  // the requested-ahead tiles are published already
      const int b0 = (int)(blockIdx.x / G);
      if (DT < 0 && !TREE && !SAMP && !P.direct && b0 < P.B) {
        const int mine = (P.NC - (int)crank + G - 1) / G;
        npre = mine < NS ? mine : NS;
        for (int i = 0; i < npre; ++i) {
          const int elem0 = ((int)crank + i * G) * C::E_TILE;
          const uint32_t bt = (uint32_t)min(C::E_TILE, P.V - elem0) * C::ST;
          const size_t rt = (size_t)b0 * (P.K + 1) * (size_t)P.V + elem0;
          mbar_expect_tx(&sm.full[i], bt);
          bulk_g2s(stages + (size_t)i * kStageBytes, P.target + rt * C::ST, bt, &sm.full[i]);
          sm.stage_parity[i] = 0;
        }
        ps = npre == NS ? 0 : npre;
        pph = npre == NS ? 1u : 0u;
        // Of the sequence's drafts these tiles need only the first (left out
        // of the sums) and their validity.  Checked here as the control warp
        // checks them when it claims the sequence (it posts exactly this job
        // then), valid rows are published at once instead of after the claim
        // -- when the CTAs (clusters) cover the batch, each verifying one
        // sequence: larger batches keep their consumers busy meanwhile.
        const bool covers = gridDim.x / (uint32_t)G >= (uint32_t)P.B;
        const int nb = !covers ? -1 : (P.draft_len ? P.draft_len[b0] : P.K);
        bool valid = covers && nb >= 0 && nb <= P.K;
        int d0 = -1;
        if (valid)
          for (int k = 0; k < nb; ++k) {
            const int32_t t = P.draft[(size_t)b0 * P.K + k];
            valid = valid && t >= 0 && t < P.V;
            if (k == 0) d0 = t;
          }
        if (valid) {
          for (int i = 0; i < npre; ++i) {
            const int c = (int)crank + i * G;
            const int elem0 = c * C::E_TILE;
            const int nel = min(C::E_TILE, P.V - elem0);
            Tag& tg = sm.tag[i];
            tg.slot = 0;
            tg.kind = kStats;
            tg.chunk = c;
            tg.nel = nel;
            tg.elem0 = elem0;
            tg.has_draft = 0;
            tg.b = b0;
            tg.j = 0;
            tg.dtok = d0;
            tg.rbase = c * kCW;
            tg.nfull = nel / C::SL;
            tg.nany = (nel + C::SL - 1) / C::SL;
            tg.dtile = d0 >= 0 ? d0 - elem0 : -1;
            tg.dwarp = (tg.dtile >= 0 && tg.dtile < nel) ? tg.dtile / C::SL : -1;
            tg.cwarps = 0;
            mbar_arrive(&sm.full[i]);  // release: the tag before the arrival
          }
          early = true;
        }
      }
      uint64_t t_idle = gtimer();
      for (;;) {
        if (vload(&sm.abort)) break;
        int si = -1, best_age = 0x7fffffff;
        for (int s = 0; s < kSlots; ++s) {
          if (vload(&sm.slot[s].state) == kReady) {
            const int a = vload(&sm.slot[s].age);
            if (a < best_age) {
              best_age = a;
              si = s;
            }
          }
        }
        if (si < 0) {
          vstore(&sm.prod_idle, 1);
          if (vload(&sm.ctrl_exited) == kSlots) break;
          if (gtimer() - t_idle > P.wait_ns) {
            set_abort(sm, G);
            break;
          }
          __nanosleep(32);
          continue;
        }
        vstore(&sm.prod_idle, 0);
        if (G > 1) fence_cluster();  // the job's words came from the cluster leader
        __threadfence_block();
        Slot& S = sm.slot[si];
        vstore(&S.state, kIssued);
        const int kind = S.kind, b = S.b, j = S.j;
        // the draft model's row is read for rows with a draft (j < n_b): its
        // statistics, and the residual pass
        const bool with_draft =
            DT >= 0 && ((kind == kStats && j < S.nb) || (kind == kResid && S.smode == 1));
        auto set_tag = [&](Tag& tg, int c) {
          const int elem0 = c * C::E_TILE;
          const int nel = min(C::E_TILE, P.V - elem0);
          tg.slot = si;
          tg.kind = kind;
          tg.chunk = c;
          tg.nel = nel;
          tg.elem0 = elem0;
          tg.has_draft = with_draft ? 1 : 0;
          tg.b = b;
          tg.j = j;
          tg.dtok = kind == kStats ? S.dtok : -1;
          tg.rbase = (si * P.NC + c) * kCW;
          tg.nfull = nel / C::SL;
          tg.nany = (nel + C::SL - 1) / C::SL;
          tg.dtile = tg.dtok >= 0 ? tg.dtok - elem0 : -1;
          tg.dwarp = (tg.dtile >= 0 && tg.dtile < nel) ? tg.dtile / C::SL : -1;
          uint32_t cw = 0;
          if (TREE && kind == kStats)
            for (int k = 0; k < S.nex; ++k) {
              const int o = S.ex[k] - elem0;
              if (o >= 0 && o < nel) cw |= 1u << (o / C::SL);
            }
          tg.cwarps = cw;
        };
        bool ok = true;
        int c_from = (int)crank;
        if (npre > 0) {
          // the tiles requested ahead: this job's if it is that row, else none
          // (published already: the job is that row, its drafts were valid)
          const bool match = early || (si == 0 && kind == kStats && b == b0 && j == 0);
          for (int i = 0; i < npre && !early; ++i) {
            if (match) set_tag(sm.tag[i], (int)crank + i * G);
            else sm.tag[i].kind = kSkip;
            mbar_arrive(&sm.full[i]);  // release: the tag before the arrival
          }
          if (match) c_from = (int)crank + npre * G;
          npre = 0;
        }
        // clusters: this CTA streams the job's tiles c = rank (mod G)
        for (int c = c_from; c < P.NC && ok; c += G) {
          const uint64_t t0 = gtimer();
          // (suspended on the barrier, not spinning: the consumers need the issue slots)
          while (!mbar_try_wait_hint(&sm.empty[ps], pph ^ 1, kSuspendNs)) {
            if (vload(&sm.abort) || gtimer() - t0 > P.wait_ns) {
              ok = false;
              break;
            }
          }
          if (!ok) break;
          const int elem0 = c * C::E_TILE;
          const int nel = min(C::E_TILE, P.V - elem0);
          set_tag(sm.tag[ps], c);
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
          set_abort(sm, G);
          break;
        }
        vstore(&sm.jobs_issued, vload(&sm.jobs_issued) + 1);
        t_idle = gtimer();
      }
      // tiles requested ahead for a job that never came: released unread (and,
      // after an abort, their copies complete the stages' phases for the drain)
      for (int i = 0; i < npre && !early; ++i) {
        sm.tag[i].kind = kSkip;
        mbar_arrive(&sm.full[i]);
      }
      if (!vload(&sm.abort)) {
        // tell the consumers to stop
        const uint64_t t0 = gtimer();
        bool ok = true;
        while (!mbar_try_wait(&sm.empty[ps], pph ^ 1)) {
          if (gtimer() - t0 > P.wait_ns) {
            ok = false;
            break;
          }
        }
        if (ok) {
          sm.tag[ps].kind = kExit;
          __threadfence_block();
          mbar_arrive(&sm.full[ps]);
        } else {
          set_abort(sm, G);
        }
      }
      if (vload(&sm.abort)) {
        atomicOr(&P.ws[2], 1u);
        // let every bulk copy this CTA issued land before the CTA exits: a
        // limit of its own, not shortened with the pipeline waits (a copy
        // still in flight after it means the memory system has failed)
        for (int s = 0; s < NS; ++s) {
          if (sm.stage_parity[s] < 0) continue;
          const uint64_t t0 = gtimer();
          while (!mbar_try_wait(&sm.full[s], (uint32_t)sm.stage_parity[s]))
            if (gtimer() - t0 > kDrainNs) break;
        }
      }
    }
  } else if (warp >= kCtrlWarp && warp < kCtrlWarp + kSlots && crank == 0) {
    // ----------------------------- control warps ----------------------------
    // One warp per sequence slot.  Slot 0 claims at once; the others wait
    // until the producer has issued this CTA's first row (every CTA of the
    // grid has started by then), so that small batches spread over all CTAs
    // while large ones keep four sequences in flight per CTA.
    const int si = warp - kCtrlWarp;
    Slot& S = sm.slot[si];
    Control<TT, DT, GREEDY, TREE, SAMP, CL> ctl(P, sm, rec, lane, si);
    int last_jobs = -1;
    uint32_t tpar = 0;  // phase parity of this slot's tile barriers for its current job
    uint64_t t_idle = gtimer();
    for (;;) {
      if (vload(&sm.abort)) break;
      const int st = __shfl_sync(kFullMask, vload(&S.state), 0);
      if (st == kEmpty) {
        // nothing left to claim (another slot found the pool empty)
        if (__shfl_sync(kFullMask, vload(&sm.pool_done), 0)) break;
        // claim when this is the CTA's first sequence, or when no row is queued
        // and the producer has issued everything (its ring covers the claim)
        int go = 0;
        if (lane == 0) {
          const bool first = si == 0 && vload(&sm.claims) == 0;
          bool want = first;
          if (!want && vload(&sm.jobs_issued) > 0) {
            // steady state: keep sequences in flight so that one streams while
            // another's decision is taken; once fewer sequences are
            // left than CTAs, claim only when the producer has run dry, so the
            // last sequences spread over the CTAs instead of queueing in few
            int busy = 0, ready = 0;
            for (int s2 = 0; s2 < kSlots; ++s2) {
              const int st2 = vload(&sm.slot[s2].state);
              busy += st2 != kEmpty;
              ready += st2 == kReady;
            }
            const bool dry = vload(&sm.prod_idle) && ready == 0;
            // decisions after sampling take longer (resample): keep more in flight
            const int target = GREEDY ? 2 : 3;
            want = dry || (busy < target && vload(&sm.pool_left) >= (int)(gridDim.x / G));
          }
          if (!want && vload(&sm.ctrl_exited) > 0) want = true;  // nothing else to wait for
          go = want && atomicCAS(&sm.claim_lock, 0, 1) == 0;
        }
        go = __shfl_sync(kFullMask, go, 0);
        if (go) {
          ctl.refill();
          __syncwarp();
          if (lane == 0) atomicExch(&sm.claim_lock, 0);
          if (!ctl.more && __shfl_sync(kFullMask, vload(&S.state), 0) == kEmpty) break;
          t_idle = gtimer();
          continue;
        }
        // an idle slot waits as long as the CTA makes progress
        int timeout = 0;
        if (lane == 0) {
          const int ji = vload(&sm.jobs_issued);
          if (ji != last_jobs) {
            last_jobs = ji;
            t_idle = gtimer();
          } else if (gtimer() - t_idle > P.wait_ns) {
            set_abort(sm, G);
            timeout = 1;
          }
        }
        if (__shfl_sync(kFullMask, timeout, 0)) break;
        __nanosleep(256);
        continue;
      }
      // a job is posted: merge its tiles as their records complete (while the
      // rest of the row streams), then decide
      bool ok = true;
      uint64_t t0 = gtimer();
      for (int c = 0; c < P.NC;) {
        // every lane waits (acquire: the tile's records are visible after it)
        const bool done = G == 1 ? mbar_try_wait(&sm.tile_bar[si][c], tpar)
                                 : mbar_try_wait_cluster(&sm.tile_bar[si][c], tpar);
        if (__all_sync(kFullMask, done)) {
          ctl.merge_tile(c);
          ++c;
          t0 = gtimer();
          continue;
        }
        int stop = 0;
        if (lane == 0) stop = vload(&sm.abort) || gtimer() - t0 > P.wait_ns;
        if (__shfl_sync(kFullMask, stop, 0)) {
          ok = false;
          break;
        }
      }
      tpar ^= 1u;  // the next job of this slot completes the next phase
      if (!ok) {
        if (lane == 0) set_abort(sm, G);
        break;
      }
      ctl.handle();
      t_idle = gtimer();
    }
    if (lane == 0) {
      if (vload(&sm.abort)) {
        // this slot's sequence, and (slot 0) any nobody will claim now: the
        // CTA's own first sequence if the abort came before its claim, and
        // the pool past the first gridDim.x
        if (S.state != kEmpty) write_result(P, S.b, -1, -1, SAMSPEC_ST_TIMEOUT);
        const uint32_t ncl = gridDim.x / (uint32_t)G;
        if (si == 0 && ctl.first_) write_result(P, (int)(blockIdx.x / G), -1, -1, SAMSPEC_ST_TIMEOUT);
        if (si == 0 && ncl < (uint32_t)P.B) {
          // under the claim lock (a slot may be claiming): unless a claim
          // already found the pool empty, claim the rest to mark them
          const uint64_t t0 = gtimer();
          bool locked = false;
          while (!(locked = atomicCAS(&sm.claim_lock, 0, 1) == 0) && gtimer() - t0 < kDrainNs) {
          }
          if (!vload(&sm.pool_done)) {
            for (uint32_t b = ncl + atomicAdd(&P.ws[0], 1u); b < (uint32_t)P.B;
                 b = ncl + atomicAdd(&P.ws[0], 1u))
              write_result(P, (int)b, -1, -1, SAMSPEC_ST_TIMEOUT);
            vstore(&sm.pool_done, 1);
          }
          end_claims(P, sm, G);
          if (locked) atomicExch(&sm.claim_lock, 0);
        }
      }
      __threadfence_block();
      atomicAdd(&sm.ctrl_exited, 1);
      // clusters: the other CTAs' producers stop once every control warp of
      // the leader has
      for (int r = 1; r < G; ++r) red_cluster_add_u32(cluster_map(&sm.ctrl_exited, (uint32_t)r), 1u);
    }
  }
  __syncthreads();
  // clusters: every store into another CTA's shared memory has landed
  // before any CTA of the cluster exits
  if (G > 1) cluster_sync_all();
  // (every CTA normally counted itself out when its claiming ended)
  if (threadIdx.x == 0) end_claims(P, sm, G);
}

__global__ void uniforms_kernel(int32_t B, int32_t K, uint64_t seed, uint64_t step, float* u) {
  const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (i >= (int64_t)B * (K + 1)) return;
  const int b = (int)(i / (K + 1)), j = (int)(i % (K + 1));
  verify_coins(seed, step, (uint32_t)b, (uint32_t)j, &u[2 * i], &u[2 * i + 1]);
}

// ---- host launch --------------------------------------------------------------
template <int TT, int DT, bool GREEDY, bool TREE = false, bool SAMP = false>
int launch(const VParams& P0, cudaStream_t stream) {
  using C = Cfg<TT, DT>;
  VParams P = P0;
  P.NC = (P.V + C::E_TILE - 1) / C::E_TILE;
  if (P.NC > (DT >= 0 ? kMaxChunksDraft : kMaxChunks)) return SAMSPEC_ESIZE;
  const size_t rec_off = (sizeof(Smem) + 15) & ~(size_t)15;
  const size_t head =
      (rec_off + rec_bytes_of<DT>(P.NC) + 1023) & ~(size_t)1023;
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
    if (cudaFuncSetAttribute(verify_kernel<TT, DT, GREEDY, TREE, SAMP>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem[dev]) !=
        cudaSuccess)
      return SAMSPEC_ECUDA;
    if constexpr (!TREE && !SAMP) {
      if (cudaFuncSetAttribute(verify_kernel<TT, DT, GREEDY, TREE, SAMP, true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem[dev]) !=
          cudaSuccess)
        return SAMSPEC_ECUDA;
    }
    attr_done[dev] = true;
  }
  int ns = (int)(((size_t)max_smem[dev] - head) / kStageBytes);
  if (ns > kMaxStages) ns = kMaxStages;
  if (ns < kMinStages) return SAMSPEC_ESIZE;
  P.NS = ns;
  P.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
  const size_t smem = head + (size_t)ns * kStageBytes;
  auto kernel = verify_kernel<TT, DT, GREEDY, TREE, SAMP>;
  auto ckernel = verify_kernel<TT, DT, GREEDY, TREE, SAMP, !TREE && !SAMP>;
  // A batch that leaves SMs idle shares each sequence's tiles among a cluster
  // of G CTAs (linear chains with bulk copies): G = 8, 4 or 2, the largest
  // with B * G CTAs on the SMs and at least two tiles per CTA of a row.
  int G = 1;
  if (!TREE && !SAMP && !P.direct)
    for (int g = 8; g >= 2; g >>= 1)
      if ((int64_t)P.B * g <= sms[dev] && P.NC >= 2 * g) {
        G = g;
        break;
      }
  int clusters = 0;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  if (G > 1) {
    cfg.gridDim = dim3((unsigned)G, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)G;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // clusters of this size resident at once (looked up once per device)
    static int max_clusters[kMaxDev][4] = {{0}};
    int& mc = max_clusters[dev][G == 2 ? 1 : (G == 4 ? 2 : 3)];
    if (mc == 0 && cudaOccupancyMaxActiveClusters(&mc, ckernel, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();
      mc = -1;
    }
    clusters = mc < P.B ? mc : P.B;
    if (clusters < 1) G = 1;
  }
  P.G = G;
  // launched with programmatic stream serialisation: the kernel's set-up
  // (shared memory, barriers) overlaps the previous kernel's tail, and
  // griddepcontrol.wait orders every global access after it
  cudaLaunchAttribute pattr[2];
  pattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pattr[0].val.programmaticStreamSerializationAllowed = 1;
  if (G == 1) {
    const int grid = P.B < sms[dev] ? P.B : sms[dev];
    cudaLaunchConfig_t c1 = {};
    c1.gridDim = dim3((unsigned)grid, 1, 1);
    c1.blockDim = dim3(kThreads, 1, 1);
    c1.dynamicSmemBytes = smem;
    c1.stream = stream;
    c1.attrs = pattr;
    c1.numAttrs = 1;
    return cudaLaunchKernelEx(&c1, kernel, P) == cudaSuccess ? SAMSPEC_OK : SAMSPEC_ECUDA;
  }
  pattr[1] = attr[0];
  cfg.attrs = pattr;
  cfg.numAttrs = 2;
  cfg.gridDim = dim3((unsigned)(clusters * G), 1, 1);
  return cudaLaunchKernelEx(&cfg, ckernel, P) == cudaSuccess ? SAMSPEC_OK : SAMSPEC_ECUDA;
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

// Scratch of spec_verify_noalloc: the kernel's three work counters (claimed
// sequences, finished CTAs, error flag), in a fixed array that every device
// loading this library holds until the process exits.
constexpr size_t kNoAllocScratchBytes = 256;
static __device__ __align__(256) uint32_t noalloc_scratch[kNoAllocScratchBytes / 4];

namespace {

// Device address of noalloc_scratch on the current device.  On the host the
// array's name only stands in for the symbol, so the address is looked up
// once per device (with that device current) and cached for the life of the
// process.  cudaDeviceReset destroys the context that address belongs to:
// after a reset of a device, this entry point must not be called on it again
// in the same process.
int noalloc_scratch_address(void** out) {
  constexpr int kMaxDev = 64;
  static std::mutex mu;
  static void* addr[kMaxDev] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return SAMSPEC_ECUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, noalloc_scratch) != cudaSuccess || !p) return SAMSPEC_ECUDA;
    addr[dev] = p;
  }
  *out = addr[dev];
  return SAMSPEC_OK;
}


// Logits per staging tile of the kernel instantiated for (target, draft)
// element types (draft -1: one-hot drafts or greedy).
int tile_elems(int tdt, int ddt) {
  if (ddt < 0) return tdt == SAMSPEC_F32 ? Cfg<0, -1>::E_TILE : Cfg<1, -1>::E_TILE;
  if (tdt == SAMSPEC_F32) return ddt == SAMSPEC_F32 ? Cfg<0, 0>::E_TILE : Cfg<0, 1>::E_TILE;
  return ddt == SAMSPEC_F32 ? Cfg<1, 0>::E_TILE : Cfg<1, 1>::E_TILE;
}

// spec_verify's host-side argument checks and kernel parameters, without the
// workspace.  Enqueues nothing; every size the kernel cannot take is refused
// here, so a caller may check before touching device memory.
int verify_params(const void* d_target, int32_t target_dtype, const void* d_draft_logits,
                  int32_t draft_dtype, const int32_t* d_draft, const int32_t* d_draft_len,
                  int32_t B, int32_t K, int32_t V, float temperature, uint64_t seed, uint64_t step,
                  int32_t* d_accept_len, int32_t* d_out_token, int32_t* d_emit,
                  int32_t* d_emit_len, int32_t* d_status, const spec_verify_debug* dbg,
                  VParams* out, int* ddt_out) {
  if (!d_target || (K > 0 && !d_draft) || !d_accept_len || !d_out_token) return SAMSPEC_EINVAL;
  if (B < 1 || B > (1 << 24) || K < 0 || K > 32 || V < 1 || V > (1 << 24)) return SAMSPEC_ESIZE;
  if (!(temperature >= 0.f) || temperature != temperature || temperature == __builtin_inff())
    return SAMSPEC_EINVAL;
  if (target_dtype != SAMSPEC_F32 && target_dtype != SAMSPEC_BF16) return SAMSPEC_EDTYPE;
  const bool greedy = temperature == 0.f;
  int ddt = -1;
  if (d_draft_logits && !greedy) {
    if (draft_dtype != SAMSPEC_F32 && draft_dtype != SAMSPEC_BF16) return SAMSPEC_EDTYPE;
    ddt = draft_dtype;
  }
  const int64_t nc = ((int64_t)V + tile_elems(target_dtype, ddt) - 1) / tile_elems(target_dtype, ddt);
  if (nc > (ddt >= 0 ? kMaxChunksDraft : kMaxChunks)) return SAMSPEC_ESIZE;
  const int st = target_dtype == SAMSPEC_F32 ? 4 : 2;
  const int sd = ddt < 0 ? 0 : (ddt == SAMSPEC_F32 ? 4 : 2);
  if (reinterpret_cast<uintptr_t>(d_target) % 16 != 0) return SAMSPEC_EALIGN;
  if (ddt >= 0 && reinterpret_cast<uintptr_t>(d_draft_logits) % 16 != 0) return SAMSPEC_EALIGN;
  VParams& P = *out;
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
  P.cTd = greedy ? 0.0 : 1.4426950408889634 / (double)temperature;
  P.cT = (float)P.cTd;
  P.cTl = (float)(P.cTd - (double)P.cT);
  P.seed = seed;
  P.step = step;
  P.accept_len = d_accept_len;
  P.out_token = d_out_token;
  P.emit = d_emit;
  P.emit_len = d_emit_len;
  P.status = d_status;
  if (dbg) P.dbg = *dbg;
  P.direct = ((size_t)V * st) % 16 != 0 || (sd && ((size_t)V * sd) % 16 != 0);
  *ddt_out = ddt;
  return SAMSPEC_OK;
}

}  // namespace

extern "C" {

size_t spec_verify_workspace_bytes(int32_t B, int32_t K, int32_t V) {
  if (B < 1 || K < 0 || V < 1) return 0;
  return kVerifyWorkspaceBytes;
}

int spec_verify_workspace_init(void* d_workspace, size_t ws_bytes, samspec_stream_t stream) {
  if (!d_workspace || ws_bytes < kVerifyWorkspaceBytes) return SAMSPEC_EINVAL;
  return cudaMemsetAsync(d_workspace, 0, kVerifyWorkspaceBytes,
                         reinterpret_cast<cudaStream_t>(stream)) ==
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
  VParams P;
  int ddt = -1;
  const int rc = verify_params(d_target, target_dtype, d_draft_logits, draft_dtype, d_draft,
                               d_draft_len, B, K, V, temperature, seed, step, d_accept_len,
                               d_out_token, d_emit, d_emit_len, d_status, dbg, &P, &ddt);
  if (rc != SAMSPEC_OK) return rc;
  if (!d_workspace) return SAMSPEC_EINVAL;
  if (ws_bytes < spec_verify_workspace_bytes(B, K, V)) return SAMSPEC_ESIZE;
  if (reinterpret_cast<uintptr_t>(d_workspace) % 256 != 0) return SAMSPEC_EALIGN;
  P.ws = static_cast<uint32_t*>(d_workspace);
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return P.T == 0.f ? dispatch<true>(P, target_dtype, ddt, s) : dispatch<false>(P, target_dtype, ddt, s);
}

size_t spec_verify_sampling_workspace_bytes(int32_t B, int32_t K, int32_t V) {
  if (B < 1 || K < 0 || V < 1) return 0;
  return 256 + (((size_t)B * (K + 1) * sizeof(float) + 255) & ~(size_t)255);
}

int spec_verify_sampling(const void* d_target, int32_t target_dtype, const int32_t* d_draft,
                         const int32_t* d_draft_len, int32_t B, int32_t K, int32_t V,
                         const float* d_temperature, const int32_t* d_top_k,
                         const float* d_top_p, uint64_t seed, uint64_t step,
                         int32_t* d_accept_len, int32_t* d_out_token, int32_t* d_emit,
                         int32_t* d_emit_len, int32_t* d_status, const spec_verify_debug* dbg,
                         void* d_workspace, size_t ws_bytes, samspec_stream_t stream) {
  if (!d_target || (K > 0 && !d_draft) || !d_temperature || !d_top_k || !d_top_p ||
      !d_accept_len || !d_out_token || !d_workspace)
    return SAMSPEC_EINVAL;
  if (B < 1 || B > (1 << 24) || K < 0 || K > 32 || V < 1) return SAMSPEC_ESIZE;
  if (target_dtype != SAMSPEC_F32 && target_dtype != SAMSPEC_BF16) return SAMSPEC_EDTYPE;
  const int st = target_dtype == SAMSPEC_F32 ? 4 : 2;
  if ((int64_t)V > (int64_t)kMaxChunks * (kStageBytes / st)) return SAMSPEC_ESIZE;
  if (ws_bytes < spec_verify_sampling_workspace_bytes(B, K, V)) return SAMSPEC_ESIZE;
  if (reinterpret_cast<uintptr_t>(d_workspace) % 256 != 0) return SAMSPEC_EALIGN;
  if (reinterpret_cast<uintptr_t>(d_target) % 16 != 0) return SAMSPEC_EALIGN;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // each row's cut, into the workspace after the kernel's counters
  float* tau = reinterpret_cast<float*>(static_cast<unsigned char*>(d_workspace) + 256);
  const int rc = launch_sampling_cut(d_target, target_dtype, B, K + 1, V, d_temperature, d_top_k,
                                     d_top_p, tau, s);
  if (rc != SAMSPEC_OK) return rc;
  VParams P;
  std::memset(&P, 0, sizeof(P));
  P.target = static_cast<const unsigned char*>(d_target);
  P.draft = d_draft;
  P.draft_len = d_draft_len;
  P.B = B;
  P.K = K;
  P.V = V;
  P.T = 1.f;  // per sequence instead (seqT)
  P.seed = seed;
  P.step = step;
  P.accept_len = d_accept_len;
  P.out_token = d_out_token;
  P.emit = d_emit;
  P.emit_len = d_emit_len;
  P.status = d_status;
  if (dbg) {
    P.dbg = *dbg;
    P.dbg.q_d = nullptr;
  }
  P.ws = static_cast<uint32_t*>(d_workspace);
  P.direct = ((size_t)V * st) % 16 != 0;
  P.seqT = d_temperature;
  P.tau = tau;
  return target_dtype == SAMSPEC_F32 ? launch<0, -1, false, false, true>(P, s)
                                     : launch<1, -1, false, false, true>(P, s);
}

int spec_verify_tree(const void* d_target, int32_t target_dtype, const int32_t* d_tok,
                     const int32_t* d_first_child, const int32_t* d_next_sibling, int32_t B,
                     int32_t N, int32_t V, float temperature, uint64_t seed, uint64_t step,
                     int32_t* d_accept_len, int32_t* d_out_token, int32_t* d_path,
                     int32_t* d_emit, int32_t* d_emit_len, int32_t* d_status,
                     const spec_verify_debug* dbg, void* d_workspace, size_t ws_bytes,
                     samspec_stream_t stream) {
  if (!d_target || !d_tok || !d_first_child || !d_next_sibling || !d_accept_len ||
      !d_out_token || !d_workspace)
    return SAMSPEC_EINVAL;
  if (B < 1 || B > (1 << 24) || N < 1 || N > 32 || V < 1 || V > (1 << 24)) return SAMSPEC_ESIZE;
  if (!(temperature >= 0.f) || temperature != temperature || temperature == __builtin_inff())
    return SAMSPEC_EINVAL;
  if (target_dtype != SAMSPEC_F32 && target_dtype != SAMSPEC_BF16) return SAMSPEC_EDTYPE;
  if (ws_bytes < spec_verify_workspace_bytes(B, N - 1, V)) return SAMSPEC_ESIZE;
  if (reinterpret_cast<uintptr_t>(d_workspace) % 256 != 0) return SAMSPEC_EALIGN;
  if (reinterpret_cast<uintptr_t>(d_target) % 16 != 0) return SAMSPEC_EALIGN;
  const bool greedy = temperature == 0.f;
  const int st = target_dtype == SAMSPEC_F32 ? 4 : 2;
  VParams P;
  std::memset(&P, 0, sizeof(P));
  P.target = static_cast<const unsigned char*>(d_target);
  P.B = B;
  P.K = N - 1;
  P.V = V;
  P.T = temperature;
  P.Td = (double)temperature;
  P.cTd = greedy ? 0.0 : 1.4426950408889634 / (double)temperature;
  P.cT = (float)P.cTd;
  P.cTl = (float)(P.cTd - (double)P.cT);
  P.seed = seed;
  P.step = step;
  P.accept_len = d_accept_len;
  P.out_token = d_out_token;
  P.emit = d_emit;
  P.emit_len = d_emit_len;
  P.status = d_status;
  if (dbg) {
    P.dbg = *dbg;
    P.dbg.p_d = nullptr;  // per-candidate probabilities are not reported for trees
    P.dbg.q_d = nullptr;
  }
  P.ws = static_cast<uint32_t*>(d_workspace);
  P.direct = ((size_t)V * st) % 16 != 0;
  P.ttok = d_tok;
  P.tfc = d_first_child;
  P.tns = d_next_sibling;
  P.path = d_path;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (greedy)
    return target_dtype == SAMSPEC_F32 ? launch<0, -1, true, true>(P, s) : launch<1, -1, true, true>(P, s);
  return target_dtype == SAMSPEC_F32 ? launch<0, -1, false, true>(P, s) : launch<1, -1, false, true>(P, s);
}

uint64_t samspec_set_wait_limit_ns(uint64_t ns) {
  return g_wait_ns.exchange(ns == 0 ? kWaitNs : ns);
}

int spec_uniforms(int32_t B, int32_t K, uint64_t seed, uint64_t step, float* d_u,
                  samspec_stream_t stream) {
  if (!d_u || B < 1 || K < 0 || K > 32) return SAMSPEC_EINVAL;
  const int64_t n = (int64_t)B * (K + 1);
  uniforms_kernel<<<(unsigned)((n + 255) / 256), 256, 0,
                    reinterpret_cast<cudaStream_t>(stream)>>>(B, K, seed, step, d_u);
  return cudaGetLastError() == cudaSuccess ? SAMSPEC_OK : SAMSPEC_ECUDA;
}

int spec_verify_noalloc(const void* d_target, int32_t target_dtype, const void* d_draft_logits,
                        int32_t draft_dtype, const int32_t* d_draft, const int32_t* d_draft_len,
                        int32_t B, int32_t K, int32_t V, float temperature, uint64_t seed,
                        uint64_t step, int32_t* d_accept_len, int32_t* d_out_token,
                        int32_t* d_emit, int32_t* d_emit_len, int32_t* d_status,
                        const spec_verify_debug* dbg, samspec_stream_t stream) {
  static_assert(kVerifyWorkspaceBytes <= kNoAllocScratchBytes, "the counters fit the scratch");
  // every argument and size is checked before anything is enqueued
  VParams P;
  int ddt = -1;
  int rc = verify_params(d_target, target_dtype, d_draft_logits, draft_dtype, d_draft, d_draft_len,
                         B, K, V, temperature, seed, step, d_accept_len, d_out_token, d_emit,
                         d_emit_len, d_status, dbg, &P, &ddt);
  if (rc != SAMSPEC_OK) return rc;
  void* ws = nullptr;
  rc = noalloc_scratch_address(&ws);
  if (rc != SAMSPEC_OK) return rc;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the counters must start at zero; the array keeps whatever the last call
  // on this device left there
  if (cudaMemsetAsync(ws, 0, kVerifyWorkspaceBytes, s) != cudaSuccess) return SAMSPEC_ECUDA;
  P.ws = static_cast<uint32_t*>(ws);
  return P.T == 0.f ? dispatch<true>(P, target_dtype, ddt, s) : dispatch<false>(P, target_dtype, ddt, s);
}

}  // extern "C"
