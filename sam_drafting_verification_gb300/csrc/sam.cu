// sam.cu -- device-resident dynamic suffix automata, one warp per sequence.
//
// Method: the D-SAM of "SAM投机推理：长序列强化学习训练加速利器" (CANN
// cann-recipes-train) §1.1 -- states are endpos classes with len / link, the
// automaton is extended by every verified token, min_endpos is kept while it is
// built, and a draft is read by walking link edges back to the first state that
// has a next edge (the ABCBC example) -- and the volcengine.com SAM-Decoding
// article §3 (Blumer's online construction; min_endpos per node; "Update of
// Suffix Automaton": extend first, then move to the matching state).
//
// GB300 layout: per sequence, struct-of-arrays regions in one caller-owned
// workspace --
//   states  int4 {len, min_endpos, tok_off, n_out | log2(tok_cap) << 24} [2C+1]
//   links   int32 suffix link per state                                  [2C+1]
//   tokens  int32 pool of per-state out-token arrays: a state's tokens sit
//           contiguously at tok_off, capacity a power of two >= 4, moved to
//           an array of twice the size when full; 4 x (3C+4) ints bound all
//           allocations
//   hash    u64 open-addressed (state, token) -> state, linear probing
//   history int32 tokens [C]
//   chain   int32 [128]: the suffix chain last, link(last), ..., root
//   scalars int32[16] {n, last, n_states, n_transitions, status, link(last),
//           len(last), token-pool top, chain length (0: not kept), 0...}
// A hash slot packs (state + 1) in bits 63..41, the token in 40..23 and the
// target state in 22..0; 0 marks an empty slot.  Slots are never deleted, so a
// key, if present, lies before the first empty slot of its probe sequence.
//
// The construction is the textbook sequential one, executed by one warp, with
// the lanes working on independent pieces of one step.  The link walk of a
// token visits the suffix chain of `last`; the warp keeps that chain in
// registers (up to 128 states), so all its (state, token) keys are probed at
// once instead of one link hop at a time: the new transitions, the out-token
// appends, the split's redirections and the next chain (the new state, then
// the distinct targets of the chain states that had the token, then the root)
// all follow from that one round of probes.  A split copies the clone's
// transitions 32 at a time.  Longer chains fall back to chasing links in
// batches of 2, 4, ... 32 states.  States are numbered in
// creation order with the new state before its clone, so the arrays equal a
// plain sequential build's.

#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include <cuda_runtime.h>

#include "common.cuh"
#include "samspec.h"

// SAMSPEC_CHECKS=1 builds the debug library: every index into a sequence's
// arrays is checked (see the element access functions below).
#ifndef SAMSPEC_CHECKS
#define SAMSPEC_CHECKS 0
#endif

struct sam_batch {
  int32_t B, C, V, S, E;
  int64_t H;
  size_t ws_bytes;
  char* ws;
  int64_t P;  // token-pool ints per sequence
  size_t off_states, off_links, off_chain, off_pool, off_hash, off_hist, off_scal;
};

namespace samspec {
namespace {

constexpr int kScal = 16;
enum { SC_N = 0, SC_LAST, SC_NS, SC_NE, SC_STATUS, SC_LINKLAST, SC_LENLAST, SC_POOL, SC_CHAIN, SC_CHECK };

// The suffix chain of `last` (last, link(last), ..., root) is kept explicitly
// while it has at most kChainMax states: 4 registers per lane inside a launch,
// kChainMax ints per sequence between launches.  SC_CHAIN holds its length,
// 0 while the chain is longer (the walk then chases links).
constexpr int kChR = 4;
constexpr int kChainMax = 32 * kChR;

// A state record: {len, min_endpos, tok_off, n_out | log2(tok_cap) << 24};
// tok_off = -1 while the state has no out-token array.  Links live in their
// own array (the walks chase them; 16 per 64-byte line).
__device__ __forceinline__ int32_t rec_nout(int4 r) { return r.w & 0xFFFFFF; }
__device__ __forceinline__ int32_t rec_cap(int4 r) { return r.z < 0 ? 0 : (1 << (r.w >> 24)); }
__device__ __forceinline__ int32_t log2_pow2(int32_t x) { return 31 - __clz(x); }

struct SeqView {
  int4* st;        // state records
  int32_t* lk;     // suffix links
  int32_t* chn;    // suffix chain of `last` between launches
  int32_t* pool;   // out-token arrays
  unsigned long long* hs;
  int32_t* hist;
  int32_t* sc;
  int32_t S, E, C, V;
  int64_t P;
  uint32_t hmask;
};

struct BatchView {
  int4* st;
  int32_t* lk;
  int32_t* chn;
  int32_t* pool;
  unsigned long long* hs;
  int32_t* hist;
  int32_t* sc;
  int32_t B, S, E, C, V;
  int64_t H, P;
};

__device__ __forceinline__ SeqView seq_view(const BatchView& v, int b) {
  SeqView s;
  s.st = v.st + (size_t)b * v.S;
  s.lk = v.lk + (size_t)b * v.S;
  s.chn = v.chn + (size_t)b * kChainMax;
  s.pool = v.pool + (size_t)b * v.P;
  s.hs = v.hs + (size_t)b * v.H;
  s.hist = v.hist + (size_t)b * v.C;
  s.sc = v.sc + (size_t)b * kScal;
  s.S = v.S;
  s.E = v.E;
  s.C = v.C;
  s.V = v.V;
  s.P = v.P;
  s.hmask = (uint32_t)(v.H - 1);
  return s;
}

// ---- element access ----------------------------------------------------------
// Every index into a sequence's arrays goes through these functions.  In the
// debug build (SAMSPEC_CHECKS=1) an index outside its array is not used: a
// read gives a neutral value, a write is dropped, and the sequence's check
// word is set; its status becomes ST_BOUNDS when the launch ends.  In the
// normal build they are plain loads and stores.
__device__ __forceinline__ bool idx_ok(const SeqView& v, int64_t i, int64_t n) {
#if SAMSPEC_CHECKS
  if (i >= 0 && i < n) return true;
  atomicOr(v.sc + SC_CHECK, 1);
  return false;
#else
  (void)v;
  (void)i;
  (void)n;
  return true;
#endif
}
__device__ __forceinline__ int4 ST(const SeqView& v, int64_t x) {
  return idx_ok(v, x, v.S) ? v.st[x] : make_int4(0, -1, -1, 0);
}
__device__ __forceinline__ void ST_W(const SeqView& v, int64_t x, int4 r) {
  if (idx_ok(v, x, v.S)) v.st[x] = r;
}
__device__ __forceinline__ int32_t LK(const SeqView& v, int64_t x) {
  return idx_ok(v, x, v.S) ? v.lk[x] : -1;
}
__device__ __forceinline__ void LK_W(const SeqView& v, int64_t x, int32_t y) {
  if (idx_ok(v, x, v.S)) v.lk[x] = y;
}
__device__ __forceinline__ int32_t POOL(const SeqView& v, int64_t i) {
  return idx_ok(v, i, v.P) ? v.pool[i] : 0;
}
__device__ __forceinline__ void POOL_W(const SeqView& v, int64_t i, int32_t t) {
  if (idx_ok(v, i, v.P)) v.pool[i] = t;
}
__device__ __forceinline__ unsigned long long HS(const SeqView& v, int64_t i) {
  return idx_ok(v, i, (int64_t)v.hmask + 1) ? v.hs[i] : 0ull;
}
__device__ __forceinline__ void HS_W(const SeqView& v, int64_t i, unsigned long long x) {
  if (idx_ok(v, i, (int64_t)v.hmask + 1)) v.hs[i] = x;
}
__device__ __forceinline__ int32_t HIST(const SeqView& v, int64_t i) {
  return idx_ok(v, i, v.C) ? v.hist[i] : -1;
}
__device__ __forceinline__ void HIST_W(const SeqView& v, int64_t i, int32_t t) {
  if (idx_ok(v, i, v.C)) v.hist[i] = t;
}
__device__ __forceinline__ int32_t CHN(const SeqView& v, int64_t i) {
  return idx_ok(v, i, kChainMax) ? v.chn[i] : -1;
}
__device__ __forceinline__ void CHN_W(const SeqView& v, int64_t i, int32_t x) {
  if (idx_ok(v, i, kChainMax)) v.chn[i] = x;
}
// the aligned 4-slot group of the hash that holds slot p (one 32-byte sector)
__device__ __forceinline__ void HS_GROUP(const SeqView& v, uint32_t p, ulonglong2& lo,
                                         ulonglong2& hi) {
  const uint32_t base = p & ~3u;
  if (!idx_ok(v, (int64_t)base + 3, (int64_t)v.hmask + 1)) {
    lo = hi = make_ulonglong2(0ull, 0ull);
    return;
  }
  const ulonglong2* gp = reinterpret_cast<const ulonglong2*>(v.hs + base);
  lo = gp[0];
  hi = gp[1];
}

__device__ __forceinline__ uint32_t slot_hash(int32_t s, int32_t t) {
  uint64_t k = ((uint64_t)(uint32_t)s << 18) | (uint32_t)t;
  k ^= k >> 33;
  k *= 0xff51afd7ed558ccdull;
  k ^= k >> 29;
  k *= 0xc4ceb9fe1a85ec53ull;
  k ^= k >> 32;
  return (uint32_t)k;
}
__device__ __forceinline__ uint64_t key_bits(int32_t s, int32_t t) {
  return ((uint64_t)(uint32_t)(s + 1) << 18) | (uint32_t)t;
}
__device__ __forceinline__ unsigned long long slot_value(int32_t s, int32_t t, int32_t to) {
  return (key_bits(s, t) << 23) | (uint32_t)to;
}

// Per-lane probe of key bits kb from slot p on: linear probing, reading the
// aligned 4-slot group (one 32-byte sector) that holds the next slot.
// Returns 1 (found: *val, *pos), 0 (absent: *pos = first empty slot of the
// probe sequence) or -1 (no empty slot in the table).
__device__ __forceinline__ int lane_probe_from(const SeqView& v, uint64_t kb, uint32_t p,
                                               uint32_t* pos, int32_t* val) {
  const uint32_t ngroups = (v.hmask >> 2) + 2;
  for (uint32_t g = 0; g < ngroups; ++g) {
    const uint32_t base = p & ~3u;
    ulonglong2 lo, hi;
    HS_GROUP(v, p, lo, hi);
    const unsigned long long x[4] = {lo.x, lo.y, hi.x, hi.y};
    const int k0 = (int)(p & 3u);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (k < k0) continue;
      if ((x[k] >> 23) == kb) {
        *pos = base + k;
        *val = (int32_t)(x[k] & 0x7FFFFFull);
        return 1;
      }
      if (x[k] == 0ull) {
        *pos = base + k;
        return 0;
      }
    }
    p = (base + 4) & v.hmask;
  }
  return -1;
}
__device__ __forceinline__ int lane_probe(const SeqView& v, int32_t s, int32_t t, uint32_t* pos,
                                          int32_t* val) {
  return lane_probe_from(v, key_bits(s, t), slot_hash(s, t) & v.hmask, pos, val);
}

// The same probe in two halves, so that several keys' first groups are in
// flight together: probe_issue loads the home group, probe_finish scans it
// and walks on only if it did not settle the key.
struct GroupLoad {
  ulonglong2 lo, hi;
  uint32_t p;
};
__device__ __forceinline__ GroupLoad probe_issue(const SeqView& v, int32_t s, int32_t t, bool on) {
  GroupLoad g;
  g.p = slot_hash(s, t) & v.hmask;
  g.lo = make_ulonglong2(0ull, 0ull);
  g.hi = g.lo;
  if (on) HS_GROUP(v, g.p, g.lo, g.hi);
  return g;
}
__device__ __forceinline__ int probe_finish(const SeqView& v, int32_t s, int32_t t,
                                            const GroupLoad& g, uint32_t* pos, int32_t* val) {
  const uint64_t kb = key_bits(s, t);
  const uint32_t base = g.p & ~3u;
  const unsigned long long x[4] = {g.lo.x, g.lo.y, g.hi.x, g.hi.y};
  const int k0 = (int)(g.p & 3u);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if (k < k0) continue;
    if ((x[k] >> 23) == kb) {
      *pos = base + k;
      *val = (int32_t)(x[k] & 0x7FFFFFull);
      return 1;
    }
    if (x[k] == 0ull) {
      *pos = base + k;
      return 0;
    }
  }
  return lane_probe_from(v, kb, (base + 4) & v.hmask, pos, val);
}

// Writes slot value `val` for the lanes with `want` set: each lane's key is
// absent and distinct from the other lanes' keys, and *pos is the first empty
// slot of its probe sequence as read before any of these writes.  Lanes that
// share a slot leave it to the lowest of them and walk on to the next empty
// slot.  Returns false if the table has no room.
__device__ __forceinline__ bool lane_place(const SeqView& v, uint32_t pos, unsigned long long val,
                                           bool want, int lane, bool known_empty = true) {
  uint32_t p = pos;  // known_empty: no write since the probe that saw p empty
  for (uint32_t i = 0; i <= v.hmask + 1; ++i) {
    if (!__any_sync(kFullMask, want)) return true;
    const uint32_t q = p & v.hmask;
    bool empty = want;
    if (want && !known_empty) empty = HS(v, q) == 0ull;
    const uint32_t key = empty ? q : (0x80000000u | (uint32_t)lane);
    const unsigned grp = __match_any_sync(kFullMask, key);
    const bool win = empty && lane == __ffs(grp) - 1;
    __syncwarp();
    if (win) HS_W(v, q, val);
    __syncwarp();
    if (win) want = false;
    known_empty = false;
    ++p;  // occupied, or taken by a lower lane: the next slot
  }
  return !__any_sync(kFullMask, want);
}

struct Scal {
  int32_t n, last, ns, ne, status, link_last, len_last, pool;
};

// Moves n tokens (n a multiple of 4; 16-byte aligned arrays) with int4 copies.
__device__ __forceinline__ void pool_move(const SeqView& v, int32_t dst, int32_t src, int32_t n,
                                          int lane) {
  if (n > 0 && !(idx_ok(v, src, v.P) && idx_ok(v, (int64_t)src + n - 1, v.P) && idx_ok(v, dst, v.P) &&
                 idx_ok(v, (int64_t)dst + n - 1, v.P)))
    return;  // (debug build: a range outside the pool; the warp leaves together)
  const int4* s4 = reinterpret_cast<const int4*>(v.pool + src);
  int4* d4 = reinterpret_cast<int4*>(v.pool + dst);
  const int32_t n4 = n >> 2;
  constexpr int U = 4;
  for (int32_t base = 0; base < n4; base += 32 * U) {
    int4 r[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int32_t k = base + u * 32 + lane;
      if (k < n4) r[u] = s4[k];
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int32_t k = base + u * 32 + lane;
      if (k < n4) d4[k] = r[u];
    }
  }
  __syncwarp();
}

// Appends token c to the out-token arrays of the states `s` of the lanes with
// `want` set (records `r` as loaded), in parallel: full arrays move to arrays
// of twice the capacity (at least 4), reserved from the pool in lane order.
// Returns a status word.
__device__ __forceinline__ int append_out(const SeqView& v, Scal& sc, int32_t s, int4 r,
                                          int32_t c, bool want, int lane) {
  const unsigned wm = __ballot_sync(kFullMask, want);
  if (!wm) return SAMSPEC_ST_OK;
  if (sc.ne + __popc(wm) > v.E) return SAMSPEC_ST_CAPACITY;
  int32_t off = r.z, n = rec_nout(r), cap = rec_cap(r);
  const bool grow = want && n == cap;
  const int32_t ncap = grow ? (cap < 4 ? 4 : 2 * cap) : 0;
  // exclusive prefix sum of the new capacities (lane order)
  int32_t incl = ncap;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_up_sync(kFullMask, incl, o);
    if (lane >= o) incl += y;
  }
  const int32_t total = __shfl_sync(kFullMask, incl, 31);
  if ((int64_t)sc.pool + total > v.P) return SAMSPEC_ST_CAPACITY;
  const int32_t noff = sc.pool + incl - ncap;
  sc.pool += total;
  // arrays that hold tokens move, one warp-wide copy each (rare)
  unsigned mv = __ballot_sync(kFullMask, grow && n > 0);
  while (mv) {
    const int l = __ffs(mv) - 1;
    mv &= mv - 1;
    pool_move(v, __shfl_sync(kFullMask, noff, l), __shfl_sync(kFullMask, off, l),
              __shfl_sync(kFullMask, n, l), lane);
  }
  if (grow) {
    off = noff;
    cap = ncap;
  }
  if (want) {
    POOL_W(v, off + n, c);
    ST_W(v, s, make_int4(r.x, r.y, off, (n + 1) | (log2_pow2(cap) << 24)));
  }
  sc.ne += __popc(wm);
  __syncwarp();
  return SAMSPEC_ST_OK;
}

// Appends token c (Blumer's online step) when the suffix chain is not kept
// (longer than kChainMax states).  Returns a status word.
//
// The link walk visits x_0 = last, x_1 = link(last), x_2, ... until a state
// with a c-transition.  It runs in batches of 2, 4, ... 32 chain states, one
// per lane: the links are chased first (cached, cheap), then every lane probes
// its own (x_j, c) and loads its record at once, so a walk of k states costs k
// link loads and about log2(k) hash round trips instead of k of each.
__device__ int extend_chase(const SeqView& v, Scal& sc, int32_t c, int lane) {
  if (c < 0 || c >= v.V) return SAMSPEC_ST_TOKEN;
  if (sc.n >= v.C || sc.ns + 2 > v.S) return SAMSPEC_ST_CAPACITY;
  const int32_t i = sc.n;
  const int32_t cur = sc.ns++;
  if (lane == 0) {
    // position i ends only suffixes of S c and exceeds every earlier end
    ST_W(v, cur, make_int4(sc.len_last + 1, i, -1, 0));
    LK_W(v, cur, -1);
    HIST_W(v, i, c);
  }
  __syncwarp();

  int guard = sc.len_last + 2;      // chain states a walk may visit
  int32_t x = sc.last;              // first chain state of the next batch
  int W = 2;
  int32_t link_cur = 0;
  int32_t p = -1, q = -1;           // the state with a c-transition and its target
  uint32_t p_pos = 0;               // slot of (p, c)
  int32_t after_p = -1;             // link(p)
  int32_t len_p = 0;
  for (;;) {
    // chain states x_j of this batch to lanes j = 0 .. m-1; `x` ends as the
    // last of them (its link is loaded below with the probes)
    int32_t mine = lane == 0 ? x : -1;
    int m = 1;
    while (m < W) {
      const int32_t y = LK(v, x);
      if (y == -1) break;
      x = y;
      if (lane == m) mine = x;
      ++m;
    }
    guard -= m;
    if (guard < 0) return SAMSPEC_ST_LOOPCAP;
    const bool has = lane < m;
    const int4 rec = has ? ST(v, mine) : make_int4(0, 0, -1, 0);
    const int32_t nx = LK(v, x);
    uint32_t pos = 0;
    int32_t val = -1;
    const int r = has ? lane_probe(v, mine, c, &pos, &val) : 0;
    if (__any_sync(kFullMask, has && r < 0)) return SAMSPEC_ST_HASHFULL;
    const unsigned fnd = __ballot_sync(kFullMask, has && r == 1);
    const int kf = fnd ? __ffs(fnd) - 1 : m;
    // (x_j, c) -> cur for the chain states before the first with a c-transition
    const bool add = has && lane < kf;
    if (!lane_place(v, pos, slot_value(mine, c, cur), add, lane)) return SAMSPEC_ST_HASHFULL;
    const int st = append_out(v, sc, mine, rec, c, add, lane);
    if (st != SAMSPEC_ST_OK) return st;
    if (fnd) {
      p = __shfl_sync(kFullMask, mine, kf);
      q = __shfl_sync(kFullMask, val, kf);
      p_pos = __shfl_sync(kFullMask, pos, kf);
      len_p = __shfl_sync(kFullMask, rec.x, kf);
      const int32_t nxt_lane = __shfl_sync(kFullMask, mine, (kf + 1) & 31);
      after_p = kf + 1 < m ? nxt_lane : nx;
      break;
    }
    if (nx == -1) break;  // the root was the last chain state: link(cur) = root
    x = nx;
    W = W < 32 ? 2 * W : 32;
  }

  if (q >= 0) {
    const int4 sq = ST(v, q);
    const int32_t lq = LK(v, q);
    if (len_p + 1 == sq.x) {
      link_cur = q;
    } else {
      // split q: the clone takes q's transitions, link and min_endpos
      if (sc.ns + 1 > v.S) return SAMSPEC_ST_CAPACITY;
      const int32_t clone = sc.ns++;
      const int32_t nq = rec_nout(sq);
      if (sc.ne + nq > v.E) return SAMSPEC_ST_CAPACITY;
      int32_t ccap = 4;
      while (ccap < nq) ccap <<= 1;
      if ((int64_t)sc.pool + ccap > v.P) return SAMSPEC_ST_CAPACITY;
      const int32_t coff = sc.pool;
      sc.pool += ccap;
      if (lane == 0) {
        ST_W(v, clone, make_int4(len_p + 1, sq.y, coff, nq | (log2_pow2(ccap) << 24)));
        LK_W(v, clone, lq);
      }
      for (int32_t base = 0; base < nq; base += 32) {
        const bool own = base + lane < nq;
        const int32_t t = own ? POOL(v, sq.z + base + lane) : 0;
        uint32_t qpos = 0, cpos = 0;
        int32_t to = -1, dummy = -1;
        const int r1 = own ? lane_probe(v, q, t, &qpos, &to) : 1;
        const int r2 = own ? lane_probe(v, clone, t, &cpos, &dummy) : 0;
        if (__any_sync(kFullMask, r1 != 1 || r2 != 0))
          return __any_sync(kFullMask, r1 < 0 || r2 < 0) ? SAMSPEC_ST_HASHFULL : SAMSPEC_ST_LOOPCAP;
        if (own) POOL_W(v, coff + base + lane, t);
        if (!lane_place(v, cpos, slot_value(clone, t, to), own, lane)) return SAMSPEC_ST_HASHFULL;
      }
      sc.ne += nq;
      // (p, c) -> clone, then the states after p on the chain while their
      // c-transition still leads to q (batched like the walk)
      if (lane == 0) HS_W(v, p_pos, slot_value(p, c, clone));
      __syncwarp();
      int32_t y = after_p;
      W = 2;
      while (y != -1) {
        int32_t mine = lane == 0 ? y : -1;
        int m = 1;
        while (m < W) {
          const int32_t z = LK(v, y);
          if (z == -1) break;
          y = z;
          if (lane == m) mine = y;
          ++m;
        }
        guard -= m;
        if (guard < 0) return SAMSPEC_ST_LOOPCAP;
        const bool has = lane < m;
        const int32_t ny = LK(v, y);
        uint32_t pos = 0;
        int32_t val = -1;
        const int r = has ? lane_probe(v, mine, c, &pos, &val) : 1;
        if (__any_sync(kFullMask, has && r < 0)) return SAMSPEC_ST_HASHFULL;
        const unsigned stop = __ballot_sync(kFullMask, has && (r == 0 || val != q));
        const int ks = stop ? __ffs(stop) - 1 : m;
        if (has && lane < ks) HS_W(v, pos, slot_value(mine, c, clone));
        __syncwarp();
        if (stop) break;
        y = ny;
        W = W < 32 ? 2 * W : 32;
      }
      if (lane == 0) LK_W(v, q, clone);
      link_cur = clone;
    }
  }
  if (lane == 0) LK_W(v, cur, link_cur);
  __syncwarp();
  sc.last = cur;
  sc.len_last += 1;
  sc.link_last = link_cur;
  sc.n += 1;
  return SAMSPEC_ST_OK;
}

template <typename T>
__device__ __forceinline__ T sel(const T (&a)[kChR], int r) {
  T x = a[0];
#pragma unroll
  for (int i = 1; i < kChR; ++i)
    if (r == i) x = a[i];
  return x;
}

// Appends token c (Blumer's online step) with the suffix chain of `last` in
// registers: lane l holds chain states l, l + 32, ... (chr), m of them.
// Every chain state's (x_j, c) key and record are fetched at once; the first
// x_k with a c-transition ends the walk (x_j, j < k, gain c -> cur); the
// targets of x_k .. x_{m-1} (q, or the clone where a split redirected them)
// are, without repeats, the suffix chain of link(cur), so the new chain is
// cur, those targets, root.  m becomes 0 if the new chain is longer than
// kChainMax.  `sh` is this warp's scratch of kChainMax + 2 ints.
__device__ int extend_chain(const SeqView& v, Scal& sc, int32_t c, int lane,
                            int32_t (&chr)[kChR], int& m, int32_t* sh) {
  if (c < 0 || c >= v.V) return SAMSPEC_ST_TOKEN;
  if (sc.n >= v.C || sc.ns + 2 > v.S) return SAMSPEC_ST_CAPACITY;
  const int32_t i = sc.n;
  const int32_t cur = sc.ns++;
  if (lane == 0) {
    // position i ends only suffixes of S c and exceeds every earlier end
    ST_W(v, cur, make_int4(sc.len_last + 1, i, -1, 0));
    LK_W(v, cur, -1);
    HIST_W(v, i, c);
  }
  bool has[kChR];
  int4 rec[kChR];
  GroupLoad gl[kChR];
#pragma unroll
  for (int r = 0; r < kChR; ++r) {
    has[r] = 32 * r + lane < m;
    rec[r] = has[r] ? ST(v, chr[r]) : make_int4(0, 0, -1, 0);
    gl[r] = probe_issue(v, chr[r], c, has[r]);
  }
  uint32_t pos[kChR];
  int32_t val[kChR];
  int pr[kChR];
#pragma unroll
  for (int r = 0; r < kChR; ++r) {
    pos[r] = 0;
    val[r] = -1;
    pr[r] = has[r] ? probe_finish(v, chr[r], c, gl[r], &pos[r], &val[r]) : 0;
  }
  bool full = false;
  int k = m;
#pragma unroll
  for (int r = 0; r < kChR; ++r) {
    full |= __any_sync(kFullMask, has[r] && pr[r] < 0);
    const unsigned f = __ballot_sync(kFullMask, has[r] && pr[r] == 1);
    if (k == m && f) k = 32 * r + __ffs(f) - 1;
  }
  if (full) return SAMSPEC_ST_HASHFULL;
  // (x_j, c) -> cur for the chain states before x_k
#pragma unroll
  for (int r = 0; r < kChR; ++r) {
    const bool want = has[r] && 32 * r + lane < k;
    if (!__any_sync(kFullMask, want)) break;
    if (!lane_place(v, pos[r], slot_value(chr[r], c, cur), want, lane, r == 0))
      return SAMSPEC_ST_HASHFULL;
    const int st = append_out(v, sc, chr[r], rec[r], c, want, lane);
    if (st != SAMSPEC_ST_OK) return st;
  }
  int32_t link_cur = 0;
  int mn = 2;  // length of the new chain
  if (k < m) {
    const int kr = k >> 5, kl = k & 31;
    const int32_t p = __shfl_sync(kFullMask, sel(chr, kr), kl);
    const int32_t q = __shfl_sync(kFullMask, sel(val, kr), kl);
    const uint32_t p_pos = __shfl_sync(kFullMask, sel(pos, kr), kl);
    int32_t lens[kChR];
#pragma unroll
    for (int r = 0; r < kChR; ++r) lens[r] = rec[r].x;
    const int32_t len_p = __shfl_sync(kFullMask, sel(lens, kr), kl);
    const int4 sq = ST(v, q);
    const int32_t lq = LK(v, q);
    int32_t clone = -1;
    if (len_p + 1 == sq.x) {
      link_cur = q;
    } else {
      // split q: the clone takes q's transitions, link and min_endpos
      if (sc.ns + 1 > v.S) return SAMSPEC_ST_CAPACITY;
      clone = sc.ns++;
      const int32_t nq = rec_nout(sq);
      if (sc.ne + nq > v.E) return SAMSPEC_ST_CAPACITY;
      int32_t ccap = 4;
      while (ccap < nq) ccap <<= 1;
      if ((int64_t)sc.pool + ccap > v.P) return SAMSPEC_ST_CAPACITY;
      const int32_t coff = sc.pool;
      sc.pool += ccap;
      if (lane == 0) {
        ST_W(v, clone, make_int4(len_p + 1, sq.y, coff, nq | (log2_pow2(ccap) << 24)));
        LK_W(v, clone, lq);
      }
      for (int32_t base = 0; base < nq; base += 32) {
        const bool own = base + lane < nq;
        const int32_t t = own ? POOL(v, sq.z + base + lane) : 0;
        uint32_t qpos = 0, cpos = 0;
        int32_t to = -1, dummy = -1;
        const int r1 = own ? lane_probe(v, q, t, &qpos, &to) : 1;
        const int r2 = own ? lane_probe(v, clone, t, &cpos, &dummy) : 0;
        if (__any_sync(kFullMask, r1 != 1 || r2 != 0))
          return __any_sync(kFullMask, r1 < 0 || r2 < 0) ? SAMSPEC_ST_HASHFULL : SAMSPEC_ST_LOOPCAP;
        if (own) POOL_W(v, coff + base + lane, t);
        if (!lane_place(v, cpos, slot_value(clone, t, to), own, lane)) return SAMSPEC_ST_HASHFULL;
      }
      sc.ne += nq;
      // every chain state from x_k on whose c-transition leads to q (a run
      // starting at x_k) now leads to the clone
#pragma unroll
      for (int r = 0; r < kChR; ++r) {
        const int j = 32 * r + lane;
        if (has[r] && j >= k && pr[r] == 1 && val[r] == q)
          HS_W(v, pos[r], slot_value(chr[r], c, clone));
      }
      (void)p;
      (void)p_pos;
      __syncwarp();
      if (lane == 0) LK_W(v, q, clone);
      link_cur = clone;
    }
    // the new chain: cur, the distinct targets of x_k .. x_{m-1}, root
    bool lost = false;
#pragma unroll
    for (int r = 0; r < kChR; ++r) lost |= has[r] && 32 * r + lane >= k && pr[r] != 1;
    if (__any_sync(kFullMask, lost)) return SAMSPEC_ST_LOOPCAP;  // a suffix without its c-transition
    int cnt = 0;
    int32_t prev_last = -1;  // target of the previous register's lane 31
#pragma unroll
    for (int r = 0; r < kChR; ++r) {
      const int j = 32 * r + lane;
      const bool in = has[r] && j >= k;
      const int32_t t = (clone >= 0 && val[r] == q) ? clone : val[r];
      int32_t prev = __shfl_up_sync(kFullMask, t, 1);
      if (lane == 0) prev = prev_last;
      const bool d = in && (j == k || t != prev);
      const unsigned dm = __ballot_sync(kFullMask, d);
      const int at = cnt + __popc(dm & ((1u << lane) - 1u)) + 1;
      if (d && at <= kChainMax) sh[at] = t;
      cnt += __popc(dm);
      prev_last = __shfl_sync(kFullMask, t, 31);
    }
    mn = cnt + 2;
  }
  if (lane == 0) {
    sh[0] = cur;
    if (mn <= kChainMax + 1) sh[mn - 1] = 0;
    LK_W(v, cur, link_cur);
  }
  __syncwarp();
  if (mn <= kChainMax) {
#pragma unroll
    for (int r = 0; r < kChR; ++r) chr[r] = 32 * r + lane < mn ? sh[32 * r + lane] : -1;
    m = mn;
  } else {
    m = 0;
  }
  __syncwarp();
  sc.last = cur;
  sc.len_last += 1;
  sc.link_last = link_cur;
  sc.n += 1;
  return SAMSPEC_ST_OK;
}

// After a chase-walk token: takes the chain up again if it is short enough
// (it has at most len(link(last)) + 2 states).
__device__ void chain_rebuild(const SeqView& v, const Scal& sc, int lane, int32_t (&chr)[kChR],
                              int& m) {
  m = 0;
  const int32_t ll = sc.link_last;
  const int32_t bound = (ll < 0 ? 0 : ST(v, ll).x) + 2;
  if (bound > kChainMax) return;
  int32_t x = sc.last;
  int n = 0;
#pragma unroll
  for (int r = 0; r < kChR; ++r) chr[r] = -1;
  while (x != -1 && n < kChainMax) {
#pragma unroll
    for (int r = 0; r < kChR; ++r)
      if (n == 32 * r + lane) chr[r] = x;
    ++n;
    x = LK(v, x);
  }
  if (x == -1) m = n;
}

__device__ void draft_one(const SeqView& v, const Scal& sc, int32_t K, int32_t* draft_row,
                          int32_t* dl_out, int32_t* ml_out, int32_t* me_out, int lane) {
  int32_t s = 0;
  int4 rec = make_int4(0, -1, -1, 0);
  if (sc.status == SAMSPEC_ST_OK && sc.n > 0) {
    // the state of S has no out-transition: start at its suffix link
    s = sc.link_last;
    int guard = sc.len_last + 1;
    while (s > 0) {
      rec = ST(v, s);
      if (rec_nout(rec) > 0) break;
      if (--guard < 0) {
        s = 0;
        break;
      }
      s = LK(v, s);
    }
    if (s < 0) s = 0;
  }
  int32_t dl = 0, ml = 0, me = -1;
  if (s > 0) {
    ml = rec.x;
    me = rec.y;
    dl = min(K, sc.n - 1 - me);
    if (dl < 0) dl = 0;
  }
  for (int t = lane; t < K; t += 32) draft_row[t] = t < dl ? HIST(v, me + 1 + t) : -1;
  if (lane == 0) {
    if (dl_out) *dl_out = dl;
    if (ml_out) *ml_out = ml;
    if (me_out) *me_out = me;
  }
}

template <bool kExtend, bool kDraft>
__global__ void __launch_bounds__(64) sam_step_kernel(BatchView bv, const int32_t* __restrict__ rows,
                                                      int32_t n_rows,
                                                      const int32_t* __restrict__ tokens,
                                                      const int32_t* __restrict__ n_new,
                                                      int32_t max_new, int32_t K, int32_t* draft,
                                                      int32_t* draft_len, int32_t* match_len,
                                                      int32_t* min_endpos) {
  // call index i (tokens, n_new and the draft outputs), automaton row b
  const int i = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (i >= n_rows) return;
  const int b = rows ? rows[i] : i;
  if (b < 0 || b >= bv.B) {  // no such automaton: an empty draft
    if (kDraft) {
      for (int t = lane; t < K; t += 32) draft[(size_t)i * K + t] = -1;
      if (lane == 0) {
        if (draft_len) draft_len[i] = 0;
        if (match_len) match_len[i] = 0;
        if (min_endpos) min_endpos[i] = -1;
      }
    }
    return;
  }
  const SeqView v = seq_view(bv, b);
  __shared__ int32_t chain_sh[2][kChainMax + 2];
  int32_t* sh = chain_sh[(threadIdx.x >> 5) & 1];
  Scal sc;
  sc.n = v.sc[SC_N];
  sc.last = v.sc[SC_LAST];
  sc.ns = v.sc[SC_NS];
  sc.ne = v.sc[SC_NE];
  sc.status = v.sc[SC_STATUS];
  sc.link_last = v.sc[SC_LINKLAST];
  sc.len_last = v.sc[SC_LENLAST];
  sc.pool = v.sc[SC_POOL];
  int m = 0;
  int32_t chr[kChR];
  if (kExtend && sc.status == SAMSPEC_ST_OK) {
    m = v.sc[SC_CHAIN];
    if (m < 0 || m > kChainMax) m = 0;
#pragma unroll
    for (int r = 0; r < kChR; ++r) chr[r] = 32 * r + lane < m ? CHN(v, 32 * r + lane) : -1;
    const int32_t nn = n_new[i];
    if (nn < 0 || nn > max_new) {
      sc.status = SAMSPEC_ST_BADDRAFT;
    } else {
      const int32_t* row = tokens + (size_t)i * max_new;
      for (int32_t base = 0; base < nn && sc.status == SAMSPEC_ST_OK; base += 32) {
        const int32_t cnt = min(32, nn - base);
        const int32_t mine = lane < cnt ? row[base + lane] : 0;
        for (int32_t k = 0; k < cnt; ++k) {
          const int32_t c = __shfl_sync(kFullMask, mine, k);
          int st;
          if (m > 0) {
            st = extend_chain(v, sc, c, lane, chr, m, sh);
          } else {
            st = extend_chase(v, sc, c, lane);
            if (st == SAMSPEC_ST_OK) chain_rebuild(v, sc, lane, chr, m);
          }
          if (st != SAMSPEC_ST_OK) {
            sc.status = st;
            break;
          }
        }
      }
    }
  }
  if (kDraft) {
    draft_one(v, sc, K, draft + (size_t)i * K, draft_len ? draft_len + i : nullptr,
              match_len ? match_len + i : nullptr, min_endpos ? min_endpos + i : nullptr, lane);
  }
#if SAMSPEC_CHECKS
  // an index that left its array in this launch freezes the sequence
  __syncwarp();
  if (v.sc[SC_CHECK] != 0) {
    if (sc.status == SAMSPEC_ST_OK) sc.status = SAMSPEC_ST_BOUNDS;
    if (!kExtend && lane == 0) v.sc[SC_STATUS] = SAMSPEC_ST_BOUNDS;
  }
#endif
  if (kExtend && lane == 0) {
    v.sc[SC_N] = sc.n;
    v.sc[SC_LAST] = sc.last;
    v.sc[SC_NS] = sc.ns;
    v.sc[SC_NE] = sc.ne;
    v.sc[SC_STATUS] = sc.status;
    v.sc[SC_LINKLAST] = sc.link_last;
    v.sc[SC_LENLAST] = sc.len_last;
    v.sc[SC_POOL] = sc.pool;
    v.sc[SC_CHAIN] = sc.status == SAMSPEC_ST_OK ? m : 0;
  }
  if (kExtend && sc.status == SAMSPEC_ST_OK) {
#pragma unroll
    for (int r = 0; r < kChR; ++r)
      if (32 * r + lane < m) CHN_W(v, 32 * r + lane, chr[r]);
  }
}

// Static use of an automaton (the volcengine.com SAM-Decoding article,
// "Drafting with Suffix Automaton" / "Update of Suffix Automaton"): automaton
// row `cb` holds a corpus and is only read; call index i follows a generated
// text with the matching state state[2i..2i+1] = {v, l} (the state of the
// longest suffix that occurs in the corpus, its length).  Each new token c
// moves it along c from v, or from the first state on v's suffix chain that
// has c (l becoming that state's len + 1), or to (root, 0).  The chain is
// walked in batches of 2, 4, ... 32 states, one per lane, probed together.
// The draft copies the K corpus tokens after min_endpos(v).
__global__ void __launch_bounds__(64) ssam_match_kernel(BatchView bv, int32_t cb, int32_t n,
                                                        int32_t* __restrict__ state,
                                                        const int32_t* __restrict__ tokens,
                                                        const int32_t* __restrict__ n_new,
                                                        int32_t max_new, int32_t K, int32_t* draft,
                                                        int32_t* draft_len, int32_t* match_len,
                                                        int32_t* min_endpos) {
  const int i = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (i >= n) return;
  const SeqView v = seq_view(bv, cb);
  const int32_t ns = v.sc[SC_NS];
  const int32_t ntext = v.sc[SC_N];
  int32_t s = state[2 * i], l = state[2 * i + 1];
  if (s < 0 || s >= ns || l < 0) {  // not a state of this automaton: start over
    s = 0;
    l = 0;
  }
  const int32_t nn = n_new ? n_new[i] : 0;
  for (int32_t t = 0; t < nn && t < max_new; ++t) {
    const int32_t c = tokens[(size_t)i * max_new + t];
    if (c < 0 || c >= v.V) {  // a token the corpus cannot hold
      s = 0;
      l = 0;
      continue;
    }
    int32_t x = s;
    int W = 2;
    bool done = false, first = true;
    int guard = v.S + 1;
    while (!done) {
      // chain states x_j of this batch to lanes j = 0 .. m-1
      int32_t mine = lane == 0 ? x : -1;
      int m = 1;
      while (m < W) {
        const int32_t y = LK(v, x);
        if (y == -1) break;
        x = y;
        if (lane == m) mine = x;
        ++m;
      }
      guard -= m;
      const bool has = lane < m;
      const int32_t len_m = has ? ST(v, mine).x : 0;
      const int32_t nx = LK(v, x);
      uint32_t pos = 0;
      int32_t val = -1;
      const int r = has ? lane_probe(v, mine, c, &pos, &val) : 0;
      const unsigned fnd = __ballot_sync(kFullMask, has && r == 1);
      if (fnd) {
        const int kf = __ffs(fnd) - 1;
        const int32_t to = __shfl_sync(kFullMask, val, kf);
        const int32_t lk = __shfl_sync(kFullMask, len_m, kf);
        // found at the current state: the match grows by one; found further
        // down the chain: the match is that state's longest string plus c
        l = (first && kf == 0) ? l + 1 : lk + 1;
        s = to;
        done = true;
      } else if (nx == -1 || guard < 0) {
        s = 0;
        l = 0;
        done = true;
      } else {
        x = nx;
        W = W < 32 ? 2 * W : 32;
        first = false;
      }
    }
  }
  if (lane == 0) {
    state[2 * i] = s;
    state[2 * i + 1] = l;
    if (match_len) match_len[i] = l;
    if (min_endpos) min_endpos[i] = s != 0 ? ST(v, s).y : -1;
  }
  int32_t dl = 0, e = -1;
  if (s != 0 && l > 0) {
    e = ST(v, s).y;
    dl = min(K, ntext - 1 - e);
    if (dl < 0) dl = 0;
  }
  for (int t = lane; t < K; t += 32) draft[(size_t)i * K + t] = t < dl ? HIST(v, e + 1 + t) : -1;
  if (lane == 0 && draft_len) draft_len[i] = dl;
#if SAMSPEC_CHECKS
  // an index that left the corpus's arrays marks the corpus automaton
  __syncwarp();
  if (lane == 0 && v.sc[SC_CHECK] != 0) v.sc[SC_STATUS] = SAMSPEC_ST_BOUNDS;
#endif
}

// Adaptive draft selection ([P4] "Drafting with Suffix Automaton"): the
// dynamic automaton's draft unless the static match is longer by more than
// l_bias.  One thread per (sequence, draft slot).
__global__ void select_drafts_kernel(int32_t n, int32_t K, const int32_t* __restrict__ dd,
                                     const int32_t* __restrict__ dl, const int32_t* __restrict__ dm,
                                     const int32_t* __restrict__ sd, const int32_t* __restrict__ sl,
                                     const int32_t* __restrict__ sm, int32_t l_bias,
                                     int32_t* __restrict__ od, int32_t* __restrict__ ol,
                                     int32_t* __restrict__ src) {
  const int64_t g = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (g >= (int64_t)n * (K + 1)) return;
  const int i = (int)(g / (K + 1)), t = (int)(g % (K + 1));
  const bool st = sm[i] > dm[i] + l_bias;
  if (t < K) {
    od[(size_t)i * K + t] = st ? sd[(size_t)i * K + t] : dd[(size_t)i * K + t];
  } else {
    ol[i] = st ? sl[i] : dl[i];
    if (src) src[i] = st ? 1 : 0;
  }
}

// Clears the hash tables of the selected sequences and empties their automata.
__global__ void sam_reset_kernel(BatchView bv, const int32_t* __restrict__ mask) {
  for (int b = blockIdx.y; b < bv.B; b += gridDim.y) {
  if (mask && mask[b] == 0) continue;
  uint4* tab = reinterpret_cast<uint4*>(bv.hs + (size_t)b * bv.H);
  const size_t n16 = (size_t)bv.H / 2;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n16;
       i += (size_t)gridDim.x * blockDim.x)
    tab[i] = make_uint4(0, 0, 0, 0);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    int32_t* sc = bv.sc + (size_t)b * kScal;
    sc[SC_N] = 0;
    sc[SC_LAST] = 0;
    sc[SC_NS] = 1;
    sc[SC_NE] = 0;
    sc[SC_STATUS] = SAMSPEC_ST_OK;
    sc[SC_LINKLAST] = -1;
    sc[SC_LENLAST] = 0;
    sc[SC_POOL] = 0;
    sc[SC_CHAIN] = 1;
    sc[SC_CHECK] = 0;
    bv.st[(size_t)b * bv.S] = make_int4(0, -1, -1, 0);
    bv.lk[(size_t)b * bv.S] = -1;
    bv.chn[(size_t)b * kChainMax] = 0;
  }
  }
}

// ---- host side --------------------------------------------------------------
constexpr int32_t kMaxB = 1 << 20;
constexpr int32_t kMaxC = (1 << 22) - 1;
constexpr int32_t kMaxV = 1 << 18;

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct Layout {
  int32_t S, E;
  int64_t H, P;
  size_t off_states, off_links, off_chain, off_pool, off_hash, off_hist, off_scal, total;
};

bool make_layout(int32_t B, int32_t C, Layout* L) {
  if (B < 1 || B > kMaxB || C < 1 || C > kMaxC) return false;
  L->S = 2 * C + 1;  // cur + clone headroom at every step
  L->E = 3 * C + 4;
  int64_t want = (int64_t)L->E + L->E / 2;
  int64_t H = 64;
  while (H < want) H <<= 1;
  L->H = H;
  // every state's arrays together stay below 4 ints per transition: a state
  // with n >= 1 out-tokens holds a final array of capacity <= max(4, 2n) and
  // left behind arrays summing to less than that
  L->P = 4 * (int64_t)L->E;
  size_t o = 0;
  L->off_states = o;
  o = align256(o + (size_t)B * L->S * sizeof(int4));
  L->off_links = o;
  o = align256(o + (size_t)B * L->S * sizeof(int32_t));
  L->off_chain = o;
  o = align256(o + (size_t)B * kChainMax * sizeof(int32_t));
  L->off_pool = o;
  o = align256(o + (size_t)B * (size_t)L->P * sizeof(int32_t));
  L->off_hash = o;
  o = align256(o + (size_t)B * (size_t)L->H * sizeof(unsigned long long));
  L->off_hist = o;
  o = align256(o + (size_t)B * C * sizeof(int32_t));
  L->off_scal = o;
  o = align256(o + (size_t)B * kScal * sizeof(int32_t));
  L->total = o;
  return true;
}

BatchView view_of(const sam_batch* s) {
  BatchView v;
  v.st = reinterpret_cast<int4*>(s->ws + s->off_states);
  v.lk = reinterpret_cast<int32_t*>(s->ws + s->off_links);
  v.chn = reinterpret_cast<int32_t*>(s->ws + s->off_chain);
  v.pool = reinterpret_cast<int32_t*>(s->ws + s->off_pool);
  v.hs = reinterpret_cast<unsigned long long*>(s->ws + s->off_hash);
  v.hist = reinterpret_cast<int32_t*>(s->ws + s->off_hist);
  v.sc = reinterpret_cast<int32_t*>(s->ws + s->off_scal);
  v.B = s->B;
  v.S = s->S;
  v.E = s->E;
  v.C = s->C;
  v.V = s->V;
  v.H = s->H;
  v.P = s->P;
  return v;
}

int launch_reset(sam_batch* s, const int32_t* mask, cudaStream_t stream) {
  const size_t n16 = (size_t)s->H / 2;
  unsigned gx = (unsigned)std::min<size_t>((n16 + 255) / 256, 64);
  if (gx == 0) gx = 1;
  dim3 grid(gx, (unsigned)std::min<int32_t>(s->B, 65535));
  sam_reset_kernel<<<grid, 256, 0, stream>>>(view_of(s), mask);
  return cudaGetLastError() == cudaSuccess ? SAMSPEC_OK : SAMSPEC_ECUDA;
}

template <bool kExtend, bool kDraft>
int launch_step(sam_batch* s, const int32_t* rows, int32_t n, const int32_t* tokens,
                const int32_t* n_new, int32_t max_new, int32_t K, int32_t* draft, int32_t* dl,
                int32_t* ml, int32_t* me, cudaStream_t stream) {
  constexpr int kWarpsPerBlock = 2;
  if (n < 1) return SAMSPEC_OK;
  const unsigned blocks = (unsigned)((n + kWarpsPerBlock - 1) / kWarpsPerBlock);
  sam_step_kernel<kExtend, kDraft><<<blocks, 32 * kWarpsPerBlock, 0, stream>>>(
      view_of(s), rows, n, tokens, n_new, max_new, K, draft, dl, ml, me);
  return cudaGetLastError() == cudaSuccess ? SAMSPEC_OK : SAMSPEC_ECUDA;
}

}  // namespace
}  // namespace samspec

using namespace samspec;

extern "C" {

size_t sam_batch_workspace_bytes(int32_t B, int32_t capacity_tokens) {
  Layout L;
  if (!make_layout(B, capacity_tokens, &L)) return 0;
  return L.total;
}

int sam_batch_create(int32_t B, int32_t capacity_tokens, int32_t vocab, void* d_workspace,
                     size_t ws_bytes, samspec_stream_t stream, sam_batch** out) {
  if (!out || !d_workspace) return SAMSPEC_EINVAL;
  *out = nullptr;
  if (vocab < 1 || vocab > kMaxV) return SAMSPEC_ESIZE;
  Layout L;
  if (!make_layout(B, capacity_tokens, &L)) return SAMSPEC_ESIZE;
  if (ws_bytes < L.total) return SAMSPEC_ESIZE;
  if (reinterpret_cast<uintptr_t>(d_workspace) % 256 != 0) return SAMSPEC_EALIGN;
  sam_batch* s = new (std::nothrow) sam_batch;
  if (!s) return SAMSPEC_EINVAL;
  s->B = B;
  s->C = capacity_tokens;
  s->V = vocab;
  s->S = L.S;
  s->E = L.E;
  s->H = L.H;
  s->P = L.P;
  s->ws_bytes = L.total;
  s->ws = static_cast<char*>(d_workspace);
  s->off_states = L.off_states;
  s->off_links = L.off_links;
  s->off_chain = L.off_chain;
  s->off_pool = L.off_pool;
  s->off_hash = L.off_hash;
  s->off_hist = L.off_hist;
  s->off_scal = L.off_scal;
  const int rc = launch_reset(s, nullptr, reinterpret_cast<cudaStream_t>(stream));
  if (rc != SAMSPEC_OK) {
    delete s;
    return rc;
  }
  *out = s;
  return SAMSPEC_OK;
}

int sam_batch_destroy(sam_batch* batch) {
  if (!batch) return SAMSPEC_EINVAL;
  delete batch;
  return SAMSPEC_OK;
}

int sam_reset(sam_batch* batch, const int32_t* d_seq_mask, samspec_stream_t stream) {
  if (!batch) return SAMSPEC_EINVAL;
  return launch_reset(batch, d_seq_mask, reinterpret_cast<cudaStream_t>(stream));
}

int sam_extend(sam_batch* batch, const int32_t* d_tokens, const int32_t* d_n_new,
               int32_t max_new, samspec_stream_t stream) {
  if (!batch || !d_n_new || max_new < 0 || (max_new > 0 && !d_tokens)) return SAMSPEC_EINVAL;
  return launch_step<true, false>(batch, nullptr, batch->B, d_tokens, d_n_new, max_new, 0,
                                  nullptr, nullptr, nullptr, nullptr,
                                  reinterpret_cast<cudaStream_t>(stream));
}

int sam_draft(sam_batch* batch, int32_t K, int32_t* d_draft, int32_t* d_draft_len,
              int32_t* d_match_len, int32_t* d_min_endpos, samspec_stream_t stream) {
  if (!batch || !d_draft) return SAMSPEC_EINVAL;
  if (K < 1 || K > 64) return SAMSPEC_ESIZE;
  return launch_step<false, true>(batch, nullptr, batch->B, nullptr, nullptr, 0, K, d_draft,
                                  d_draft_len, d_match_len, d_min_endpos,
                                  reinterpret_cast<cudaStream_t>(stream));
}

int sam_step(sam_batch* batch, const int32_t* d_tokens, const int32_t* d_n_new, int32_t max_new,
             int32_t K, int32_t* d_draft, int32_t* d_draft_len, int32_t* d_match_len,
             int32_t* d_min_endpos, samspec_stream_t stream) {
  if (!batch || !d_n_new || !d_draft || max_new < 0 || (max_new > 0 && !d_tokens))
    return SAMSPEC_EINVAL;
  if (K < 1 || K > 64) return SAMSPEC_ESIZE;
  return launch_step<true, true>(batch, nullptr, batch->B, d_tokens, d_n_new, max_new, K,
                                 d_draft, d_draft_len, d_match_len, d_min_endpos,
                                 reinterpret_cast<cudaStream_t>(stream));
}

int sam_step_rows(sam_batch* batch, const int32_t* d_rows, int32_t n, const int32_t* d_tokens,
                  const int32_t* d_n_new, int32_t max_new, int32_t K, int32_t* d_draft,
                  int32_t* d_draft_len, int32_t* d_match_len, int32_t* d_min_endpos,
                  samspec_stream_t stream) {
  if (!batch || n < 0 || (n > 0 && !d_n_new) || max_new < 0 || (max_new > 0 && !d_tokens))
    return SAMSPEC_EINVAL;
  if (!d_rows && n > batch->B) return SAMSPEC_ESIZE;
  if (K < 0 || K > 64) return SAMSPEC_ESIZE;
  if (K > 0 && !d_draft) return SAMSPEC_EINVAL;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (K == 0) {
    // no draft: draft_len reads 0 for every sequence of the call
    if (d_draft_len && n > 0 &&
        cudaMemsetAsync(d_draft_len, 0, (size_t)n * sizeof(int32_t), st) != cudaSuccess)
      return SAMSPEC_ECUDA;
    return launch_step<true, false>(batch, d_rows, n, d_tokens, d_n_new, max_new, 0, nullptr,
                                    nullptr, nullptr, nullptr, st);
  }
  return launch_step<true, true>(batch, d_rows, n, d_tokens, d_n_new, max_new, K, d_draft,
                                 d_draft_len, d_match_len, d_min_endpos, st);
}

int ssam_match(const sam_batch* corpus, int32_t corpus_row, int32_t n, int32_t* d_state,
               const int32_t* d_tokens, const int32_t* d_n_new, int32_t max_new, int32_t K,
               int32_t* d_draft, int32_t* d_draft_len, int32_t* d_match_len,
               int32_t* d_min_endpos, samspec_stream_t stream) {
  if (!corpus || !d_state || n < 0 || max_new < 0 || (max_new > 0 && (!d_tokens || !d_n_new)) ||
      (K > 0 && !d_draft))
    return SAMSPEC_EINVAL;
  if (corpus_row < 0 || corpus_row >= corpus->B || K < 0 || K > 64) return SAMSPEC_ESIZE;
  if (n == 0) return SAMSPEC_OK;
  constexpr int kWarpsPerBlock = 2;
  const unsigned blocks = (unsigned)((n + kWarpsPerBlock - 1) / kWarpsPerBlock);
  ssam_match_kernel<<<blocks, 32 * kWarpsPerBlock, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      view_of(corpus), corpus_row, n, d_state, d_tokens, max_new > 0 ? d_n_new : nullptr, max_new,
      K, d_draft, d_draft_len, d_match_len, d_min_endpos);
  return cudaGetLastError() == cudaSuccess ? SAMSPEC_OK : SAMSPEC_ECUDA;
}

int sam_select_drafts(int32_t n, int32_t K, const int32_t* d_dyn_draft, const int32_t* d_dyn_len,
                      const int32_t* d_dyn_match, const int32_t* d_st_draft,
                      const int32_t* d_st_len, const int32_t* d_st_match, int32_t l_bias,
                      int32_t* d_draft, int32_t* d_draft_len, int32_t* d_source,
                      samspec_stream_t stream) {
  if (n < 0 || K < 0 || K > 64) return SAMSPEC_ESIZE;
  if (n == 0) return SAMSPEC_OK;
  if (!d_dyn_len || !d_dyn_match || !d_st_len || !d_st_match || !d_draft_len ||
      (K > 0 && (!d_dyn_draft || !d_st_draft || !d_draft)))
    return SAMSPEC_EINVAL;
  const int64_t total = (int64_t)n * (K + 1);
  select_drafts_kernel<<<(unsigned)((total + 255) / 256), 256, 0,
                         reinterpret_cast<cudaStream_t>(stream)>>>(
      n, K, d_dyn_draft, d_dyn_len, d_dyn_match, d_st_draft, d_st_len, d_st_match, l_bias, d_draft,
      d_draft_len, d_source);
  return cudaGetLastError() == cudaSuccess ? SAMSPEC_OK : SAMSPEC_ECUDA;
}

int sam_get_status(sam_batch* batch, int32_t* h_status, samspec_stream_t stream) {
  if (!batch || !h_status) return SAMSPEC_EINVAL;
  std::vector<int32_t> tmp((size_t)batch->B * kScal);
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(tmp.data(), batch->ws + batch->off_scal, tmp.size() * sizeof(int32_t),
                      cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return SAMSPEC_ECUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return SAMSPEC_ECUDA;
  for (int32_t b = 0; b < batch->B; ++b) h_status[b] = tmp[(size_t)b * kScal + SC_STATUS];
  return SAMSPEC_OK;
}

int sam_export(sam_batch* batch, void* d_dst, size_t bytes, samspec_stream_t stream) {
  if (!batch || !d_dst) return SAMSPEC_EINVAL;
  if (bytes < batch->ws_bytes) return SAMSPEC_ESIZE;
  return cudaMemcpyAsync(d_dst, batch->ws, batch->ws_bytes, cudaMemcpyDeviceToDevice,
                         reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? SAMSPEC_OK
             : SAMSPEC_ECUDA;
}

int sam_import(sam_batch* batch, const void* d_src, size_t bytes, samspec_stream_t stream) {
  if (!batch || !d_src) return SAMSPEC_EINVAL;
  if (bytes < batch->ws_bytes) return SAMSPEC_ESIZE;
  return cudaMemcpyAsync(batch->ws, d_src, batch->ws_bytes, cudaMemcpyDeviceToDevice,
                         reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? SAMSPEC_OK
             : SAMSPEC_ECUDA;
}

int sam_dump_sequence(sam_batch* batch, int32_t b, int32_t* h_scalars, int32_t* h_len,
                      int32_t* h_link, int32_t* h_min_endpos, int32_t max_states,
                      int32_t* h_edges, int32_t max_edges, samspec_stream_t stream) {
  if (!batch || b < 0 || b >= batch->B || max_states < 0 || max_edges < 0) return SAMSPEC_EINVAL;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int32_t sc[kScal];
  const BatchView v = view_of(batch);
  if (cudaMemcpyAsync(sc, v.sc + (size_t)b * kScal, sizeof(sc), cudaMemcpyDeviceToHost, st) !=
          cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return SAMSPEC_ECUDA;
  if (h_scalars) std::memcpy(h_scalars, sc, 8 * sizeof(int32_t));
  const int32_t ns = std::min(sc[SC_NS], batch->S);
  std::vector<int4> states((size_t)ns);
  std::vector<int32_t> links((size_t)ns);
  std::vector<unsigned long long> tab((size_t)batch->H);
  if (cudaMemcpyAsync(states.data(), v.st + (size_t)b * batch->S, (size_t)ns * sizeof(int4),
                      cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaMemcpyAsync(links.data(), v.lk + (size_t)b * batch->S, (size_t)ns * sizeof(int32_t),
                      cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaMemcpyAsync(tab.data(), v.hs + (size_t)b * batch->H, tab.size() * sizeof(tab[0]),
                      cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return SAMSPEC_ECUDA;
  for (int32_t i = 0; i < ns && i < max_states; ++i) {
    if (h_len) h_len[i] = states[i].x;
    if (h_link) h_link[i] = links[i];
    if (h_min_endpos) h_min_endpos[i] = states[i].y;
  }
  if (h_edges) {
    std::vector<int64_t> keys;
    for (unsigned long long x : tab) {
      if (!x) continue;
      const int64_t s = (int64_t)(x >> 41) - 1, t = (int64_t)((x >> 23) & 0x3FFFF),
                    to = (int64_t)(x & 0x7FFFFF);
      keys.push_back((s << 41) | (t << 23) | to);
    }
    std::sort(keys.begin(), keys.end());
    for (size_t e = 0; e < keys.size() && (int64_t)e < max_edges; ++e) {
      h_edges[3 * e + 0] = (int32_t)(keys[e] >> 41);
      h_edges[3 * e + 1] = (int32_t)((keys[e] >> 23) & 0x3FFFF);
      h_edges[3 * e + 2] = (int32_t)(keys[e] & 0x7FFFFF);
    }
  }
  return SAMSPEC_OK;
}

}  // extern "C"
