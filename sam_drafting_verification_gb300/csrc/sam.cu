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
//   states  int4 {len, link, min_endpos, edge_head}   [2C+1]
//   edges   int2 {token, next}  (per-state out-transition lists) [3C+4]
//   hash    u64 open-addressed (state, token) -> state, linear probing,
//           probed 32 slots at a time by the whole warp (one 256-byte window)
//   history int32 tokens [C]
//   scalars int32[8] {n, last, n_states, n_edges, status, link(last),
//           len(last), 0}
// A hash slot packs (state + 1) in bits 63..41, the token in 40..23 and the
// target state in 22..0; 0 marks an empty slot.  Slots are never deleted, so a
// key, if present, lies before the first empty slot of its probe sequence.
//
// The construction is the textbook sequential one, executed by one warp:
// every lane runs the same scalar control flow, and the lanes cooperate only in
// the 32-slot hash probes.  States are numbered in creation order with the new
// state before its clone, so the arrays equal a plain sequential build's.

#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include <cuda_runtime.h>

#include "common.cuh"
#include "samspec.h"

struct sam_batch {
  int32_t B, C, V, S, E;
  int64_t H;
  size_t ws_bytes;
  char* ws;
  size_t off_states, off_edges, off_hash, off_hist, off_scal;
};

namespace samspec {
namespace {

constexpr int kScal = 8;
enum { SC_N = 0, SC_LAST, SC_NS, SC_NE, SC_STATUS, SC_LINKLAST, SC_LENLAST };

struct SeqView {
  int4* st;
  int2* ed;
  unsigned long long* hs;
  int32_t* hist;
  int32_t* sc;
  int32_t S, E, C, V;
  uint32_t hmask;
  uint32_t nwin;  // number of 32-slot windows in the table
};

struct BatchView {
  int4* st;
  int2* ed;
  unsigned long long* hs;
  int32_t* hist;
  int32_t* sc;
  int32_t B, S, E, C, V;
  int64_t H;
};

__device__ __forceinline__ SeqView seq_view(const BatchView& v, int b) {
  SeqView s;
  s.st = v.st + (size_t)b * v.S;
  s.ed = v.ed + (size_t)b * v.E;
  s.hs = v.hs + (size_t)b * v.H;
  s.hist = v.hist + (size_t)b * v.C;
  s.sc = v.sc + (size_t)b * kScal;
  s.S = v.S;
  s.E = v.E;
  s.C = v.C;
  s.V = v.V;
  s.hmask = (uint32_t)(v.H - 1);
  s.nwin = (uint32_t)(v.H / 32);
  return s;
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

// Warp-cooperative probe of (s, t).  Returns 1 (found: *pos, *val), 0 (absent:
// *pos = first empty slot of the probe sequence) or -1 (table full).
__device__ __forceinline__ int probe(const SeqView& v, int32_t s, int32_t t, uint32_t* pos,
                                     int32_t* val, int lane) {
  const uint64_t kb = key_bits(s, t);
  const uint32_t h = slot_hash(s, t);
  for (uint32_t w = 0; w < v.nwin; ++w) {
    const uint32_t p = (h + w * 32u + (uint32_t)lane) & v.hmask;
    const unsigned long long x = v.hs[p];
    const unsigned m = __ballot_sync(kFullMask, (x >> 23) == kb);
    if (m) {
      const int src = __ffs(m) - 1;
      *pos = __shfl_sync(kFullMask, p, src);
      *val = (int32_t)(__shfl_sync(kFullMask, x, src) & 0x7FFFFFull);
      return 1;
    }
    const unsigned e = __ballot_sync(kFullMask, x == 0ull);
    if (e) {
      *pos = __shfl_sync(kFullMask, p, __ffs(e) - 1);
      return 0;
    }
  }
  return -1;
}

__device__ __forceinline__ void hash_write(const SeqView& v, uint32_t pos, int32_t s, int32_t t,
                                           int32_t to, int lane) {
  if (lane == 0) v.hs[pos] = (key_bits(s, t) << 23) | (uint32_t)to;
  __syncwarp();
}

struct Scal {
  int32_t n, last, ns, ne, status, link_last, len_last;
};

// Adds token t to state s's out-transition list (head = current list head).
__device__ __forceinline__ bool add_edge(const SeqView& v, Scal& sc, int32_t s, int32_t t,
                                         int32_t head, int lane) {
  if (sc.ne >= v.E) return false;
  const int32_t e = sc.ne++;
  if (lane == 0) {
    v.ed[e] = make_int2(t, head);
    reinterpret_cast<int32_t*>(&v.st[s])[3] = e;
  }
  __syncwarp();
  return true;
}

// Plain loads: every write to a sequence's arrays is made by the lanes of the
// same warp and ordered by __syncwarp(), which is also a compiler barrier.
__device__ __forceinline__ int4 load_state(const SeqView& v, int32_t s) { return v.st[s]; }

// Appends token c (Blumer's online step).  Returns a status word.
__device__ int extend_one(const SeqView& v, Scal& sc, int32_t c, int lane) {
  if (c < 0 || c >= v.V) return SAMSPEC_ST_TOKEN;
  if (sc.n >= v.C || sc.ns + 2 > v.S) return SAMSPEC_ST_CAPACITY;
  const int32_t i = sc.n;
  const int32_t cur = sc.ns++;
  if (lane == 0) {
    // position i ends only suffixes of S c and exceeds every earlier end
    v.st[cur] = make_int4(sc.len_last + 1, -1, i, -1);
    v.hist[i] = c;
  }
  __syncwarp();
  uint32_t pos;
  int32_t val;
  // `last` never has an out-transition, so (last, c) is absent
  int r = probe(v, sc.last, c, &pos, &val, lane);
  if (r < 0) return SAMSPEC_ST_HASHFULL;
  if (r > 0) return SAMSPEC_ST_LOOPCAP;
  hash_write(v, pos, sc.last, c, cur, lane);
  if (!add_edge(v, sc, sc.last, c, -1, lane)) return SAMSPEC_ST_CAPACITY;

  int32_t p = sc.link_last;
  int32_t link_cur = 0;
  int guard = sc.len_last + 2;
  for (;;) {
    if (p == -1) {
      link_cur = 0;
      break;
    }
    if (--guard < 0) return SAMSPEC_ST_LOOPCAP;
    const int4 sp = load_state(v, p);  // issued together with the probe's window
    r = probe(v, p, c, &pos, &val, lane);
    if (r < 0) return SAMSPEC_ST_HASHFULL;
    if (r == 0) {
      hash_write(v, pos, p, c, cur, lane);
      if (!add_edge(v, sc, p, c, sp.w, lane)) return SAMSPEC_ST_CAPACITY;
      p = sp.y;
      continue;
    }
    const int32_t q = val;
    const int4 sq = load_state(v, q);
    if (sp.x + 1 == sq.x) {
      link_cur = q;
      break;
    }
    // split q: the clone copies q's transitions, link and min_endpos
    if (sc.ns + 1 > v.S) return SAMSPEC_ST_CAPACITY;
    const int32_t clone = sc.ns++;
    if (lane == 0) v.st[clone] = make_int4(sp.x + 1, sq.y, sq.z, -1);
    __syncwarp();
    int32_t e = sq.w;
    int32_t clone_head = -1;
    int eguard = v.E + 1;
    while (e != -1) {
      if (--eguard < 0) return SAMSPEC_ST_LOOPCAP;
      const int2 ed = v.ed[e];
      int32_t to;
      uint32_t qpos;
      r = probe(v, q, ed.x, &qpos, &to, lane);
      if (r != 1) return r < 0 ? SAMSPEC_ST_HASHFULL : SAMSPEC_ST_LOOPCAP;
      uint32_t cpos;
      int32_t dummy;
      r = probe(v, clone, ed.x, &cpos, &dummy, lane);
      if (r != 0) return r < 0 ? SAMSPEC_ST_HASHFULL : SAMSPEC_ST_LOOPCAP;
      hash_write(v, cpos, clone, ed.x, to, lane);
      if (sc.ne >= v.E) return SAMSPEC_ST_CAPACITY;
      const int32_t ne = sc.ne++;
      if (lane == 0) v.ed[ne] = make_int2(ed.x, clone_head);
      __syncwarp();
      clone_head = ne;
      e = ed.y;
    }
    if (lane == 0) reinterpret_cast<int32_t*>(&v.st[clone])[3] = clone_head;
    // redirect (p', c) -> q to the clone along p's suffix links
    hash_write(v, pos, p, c, clone, lane);
    int32_t pp = sp.y;
    while (pp != -1) {
      if (--guard < 0) return SAMSPEC_ST_LOOPCAP;
      const int4 spp = load_state(v, pp);
      uint32_t ppos;
      int32_t pval;
      r = probe(v, pp, c, &ppos, &pval, lane);
      if (r < 0) return SAMSPEC_ST_HASHFULL;
      if (r == 0 || pval != q) break;
      hash_write(v, ppos, pp, c, clone, lane);
      pp = spp.y;
    }
    if (lane == 0) reinterpret_cast<int32_t*>(&v.st[q])[1] = clone;
    link_cur = clone;
    break;
  }
  if (lane == 0) reinterpret_cast<int32_t*>(&v.st[cur])[1] = link_cur;
  __syncwarp();
  sc.last = cur;
  sc.len_last += 1;
  sc.link_last = link_cur;
  sc.n += 1;
  return SAMSPEC_ST_OK;
}

__device__ void draft_one(const SeqView& v, const Scal& sc, int32_t K, int32_t* draft_row,
                          int32_t* dl_out, int32_t* ml_out, int32_t* me_out, int lane) {
  int32_t s = 0;
  int4 rec = make_int4(0, -1, -1, -1);
  if (sc.status == SAMSPEC_ST_OK && sc.n > 0) {
    // the state of S has no out-transition: start at its suffix link
    s = sc.link_last;
    int guard = sc.len_last + 1;
    while (s > 0) {
      rec = load_state(v, s);
      if (rec.w != -1) break;
      if (--guard < 0) {
        s = 0;
        break;
      }
      s = rec.y;
    }
    if (s < 0) s = 0;
  }
  int32_t dl = 0, ml = 0, me = -1;
  if (s > 0) {
    ml = rec.x;
    me = rec.z;
    dl = min(K, sc.n - 1 - me);
    if (dl < 0) dl = 0;
  }
  for (int t = lane; t < K; t += 32) draft_row[t] = t < dl ? v.hist[me + 1 + t] : -1;
  if (lane == 0) {
    if (dl_out) *dl_out = dl;
    if (ml_out) *ml_out = ml;
    if (me_out) *me_out = me;
  }
}

template <bool kExtend, bool kDraft>
__global__ void __launch_bounds__(64) sam_step_kernel(BatchView bv, const int32_t* __restrict__ tokens,
                                                      const int32_t* __restrict__ n_new,
                                                      int32_t max_new, int32_t K, int32_t* draft,
                                                      int32_t* draft_len, int32_t* match_len,
                                                      int32_t* min_endpos) {
  const int b = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= bv.B) return;
  const SeqView v = seq_view(bv, b);
  Scal sc;
  sc.n = v.sc[SC_N];
  sc.last = v.sc[SC_LAST];
  sc.ns = v.sc[SC_NS];
  sc.ne = v.sc[SC_NE];
  sc.status = v.sc[SC_STATUS];
  sc.link_last = v.sc[SC_LINKLAST];
  sc.len_last = v.sc[SC_LENLAST];
  if (kExtend && sc.status == SAMSPEC_ST_OK) {
    const int32_t nn = n_new[b];
    if (nn < 0 || nn > max_new) {
      sc.status = SAMSPEC_ST_BADDRAFT;
    } else {
      const int32_t* row = tokens + (size_t)b * max_new;
      for (int32_t base = 0; base < nn && sc.status == SAMSPEC_ST_OK; base += 32) {
        const int32_t cnt = min(32, nn - base);
        const int32_t mine = lane < cnt ? row[base + lane] : 0;
        for (int32_t k = 0; k < cnt; ++k) {
          const int32_t c = __shfl_sync(kFullMask, mine, k);
          const int st = extend_one(v, sc, c, lane);
          if (st != SAMSPEC_ST_OK) {
            sc.status = st;
            break;
          }
        }
      }
    }
  }
  if (kDraft) {
    draft_one(v, sc, K, draft + (size_t)b * K, draft_len ? draft_len + b : nullptr,
              match_len ? match_len + b : nullptr, min_endpos ? min_endpos + b : nullptr, lane);
  }
  if (kExtend && lane == 0) {
    v.sc[SC_N] = sc.n;
    v.sc[SC_LAST] = sc.last;
    v.sc[SC_NS] = sc.ns;
    v.sc[SC_NE] = sc.ne;
    v.sc[SC_STATUS] = sc.status;
    v.sc[SC_LINKLAST] = sc.link_last;
    v.sc[SC_LENLAST] = sc.len_last;
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
    sc[7] = 0;
    bv.st[(size_t)b * bv.S] = make_int4(0, -1, -1, -1);
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
  int64_t H;
  size_t off_states, off_edges, off_hash, off_hist, off_scal, total;
};

bool make_layout(int32_t B, int32_t C, Layout* L) {
  if (B < 1 || B > kMaxB || C < 1 || C > kMaxC) return false;
  L->S = 2 * C + 1;  // cur + clone headroom at every step
  L->E = 3 * C + 4;
  int64_t want = (int64_t)L->E + L->E / 2;
  int64_t H = 64;
  while (H < want) H <<= 1;
  L->H = H;
  size_t o = 0;
  L->off_states = o;
  o = align256(o + (size_t)B * L->S * sizeof(int4));
  L->off_edges = o;
  o = align256(o + (size_t)B * L->E * sizeof(int2));
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
  v.ed = reinterpret_cast<int2*>(s->ws + s->off_edges);
  v.hs = reinterpret_cast<unsigned long long*>(s->ws + s->off_hash);
  v.hist = reinterpret_cast<int32_t*>(s->ws + s->off_hist);
  v.sc = reinterpret_cast<int32_t*>(s->ws + s->off_scal);
  v.B = s->B;
  v.S = s->S;
  v.E = s->E;
  v.C = s->C;
  v.V = s->V;
  v.H = s->H;
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
int launch_step(sam_batch* s, const int32_t* tokens, const int32_t* n_new, int32_t max_new,
                int32_t K, int32_t* draft, int32_t* dl, int32_t* ml, int32_t* me,
                cudaStream_t stream) {
  constexpr int kWarpsPerBlock = 2;
  const unsigned blocks = (unsigned)((s->B + kWarpsPerBlock - 1) / kWarpsPerBlock);
  sam_step_kernel<kExtend, kDraft><<<blocks, 32 * kWarpsPerBlock, 0, stream>>>(
      view_of(s), tokens, n_new, max_new, K, draft, dl, ml, me);
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
  s->ws_bytes = L.total;
  s->ws = static_cast<char*>(d_workspace);
  s->off_states = L.off_states;
  s->off_edges = L.off_edges;
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
  return launch_step<true, false>(batch, d_tokens, d_n_new, max_new, 0, nullptr, nullptr,
                                  nullptr, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

int sam_draft(sam_batch* batch, int32_t K, int32_t* d_draft, int32_t* d_draft_len,
              int32_t* d_match_len, int32_t* d_min_endpos, samspec_stream_t stream) {
  if (!batch || !d_draft) return SAMSPEC_EINVAL;
  if (K < 1 || K > 64) return SAMSPEC_ESIZE;
  return launch_step<false, true>(batch, nullptr, nullptr, 0, K, d_draft, d_draft_len,
                                  d_match_len, d_min_endpos,
                                  reinterpret_cast<cudaStream_t>(stream));
}

int sam_step(sam_batch* batch, const int32_t* d_tokens, const int32_t* d_n_new, int32_t max_new,
             int32_t K, int32_t* d_draft, int32_t* d_draft_len, int32_t* d_match_len,
             int32_t* d_min_endpos, samspec_stream_t stream) {
  if (!batch || !d_n_new || !d_draft || max_new < 0 || (max_new > 0 && !d_tokens))
    return SAMSPEC_EINVAL;
  if (K < 1 || K > 64) return SAMSPEC_ESIZE;
  return launch_step<true, true>(batch, d_tokens, d_n_new, max_new, K, d_draft, d_draft_len,
                                 d_match_len, d_min_endpos,
                                 reinterpret_cast<cudaStream_t>(stream));
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
  if (h_scalars) std::memcpy(h_scalars, sc, sizeof(sc));
  const int32_t ns = std::min(sc[SC_NS], batch->S);
  std::vector<int4> states((size_t)ns);
  std::vector<unsigned long long> tab((size_t)batch->H);
  if (cudaMemcpyAsync(states.data(), v.st + (size_t)b * batch->S, (size_t)ns * sizeof(int4),
                      cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaMemcpyAsync(tab.data(), v.hs + (size_t)b * batch->H, tab.size() * sizeof(tab[0]),
                      cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return SAMSPEC_ECUDA;
  for (int32_t i = 0; i < ns && i < max_states; ++i) {
    if (h_len) h_len[i] = states[i].x;
    if (h_link) h_link[i] = states[i].y;
    if (h_min_endpos) h_min_endpos[i] = states[i].z;
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
