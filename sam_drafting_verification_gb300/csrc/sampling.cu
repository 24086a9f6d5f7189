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
// Two kernels find tau exactly.
//
// bf16 rows (cut_hist_kernel): a count per bit pattern in shared memory, one
// streaming pass per row; the cuts follow from the counts and from fixed-point
// masses computed once per non-empty pattern (details above that kernel).
//
// fp32 rows, and bf16 rows whose 16-bit counts wrap (cut_kernel, one CTA of
// 256 threads per row): the row maximum; counts and approximate masses in
// 1,024 log-scale bins of the term; the logits of the bins that hold the cuts
// copied to shared memory and sorted.  Where those bins hold too many logits,
// radix selection over order-preserving 32-bit keys of the logits (8-bit
// digits from the top: two levels for bf16 rows, whose low 16 key bits are
// fixed by the sign, four for fp32): each level streams the row and builds a
// 256-bin histogram of counts and masses of the keys that share the prefix
// chosen so far; one warp then scans the bins from the top for the digit where
// the running count reaches k (or the running mass reaches top_p * Z_k).
// Masses there are 2^(l log2(e)/T - R) in fixed point (units of 2^-42, R =
// ceil(max l log2(e)/T)) summed with integer atomics, so the sums are exact
// and the result does not depend on the order of the additions; lanes of a
// warp that hit the same bin are combined first.  Terms below 2^-43 of the
// row's maximum are dropped (at V = 2^21 at most 2^-21 of the mass).

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
constexpr int kMaxV = 1 << 21;          // keeps every mass sum below 2^63 (terms <= 2^42)

// Order-preserving key of a logit: key(a) < key(b) iff a < b, equal iff
// a == b (-0 is folded into +0 first).
__device__ __forceinline__ uint32_t order_key(float x) {
  const uint32_t u = __float_as_uint(x + 0.f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

constexpr int kLogBins = 1024;  // 32 per octave of the term, 32 octaves
constexpr int kCap = 4096;     // boundary logits held in shared memory (a power of two:
                               // the sort pads to one)

struct CutSmem {
  // radix levels over keys (the path for rows whose boundary bins overflow)
  uint32_t cnt[kBins];
  unsigned long long mass[kBins];
  // log-scale bins of the term 2^(l cT - R): exact counts, and masses
  // relative to each bin's centre in units of 2^-10 (lmassr; about 1e-3
  // accurate: they only choose which bins to collect), turned into fp32
  // masses (lmass) before the scans
  uint32_t lcnt[kLogBins];
  uint32_t lmassr[kLogBins];
  float lmass[kLogBins];
  // the logits of the boundary bins: keys and terms
  uint32_t bkey[kCap];
  float bmass[kCap];
  double tsum[kThr];  // per-thread partial sums
  float red[kThr / 32];
  uint32_t nbuf;
  uint32_t idx;
  // broadcast of warp 0's choices
  uint32_t dlo, dhi, nrange, above_in_range;
  uint32_t key;
  double dscr[4];  // broadcast scratch
};

// Log-scale bin of y = l cT - R <= ~0: b = round(-32 y) clamped to
// [0, kLogBins - 1] (32 bins per octave of the term 2^y, the last holding
// everything below about 2^-32), returned as the digit kLogBins - 1 - b
// (higher = larger logit) and as the float bf = b.  The rounding goes through
// the 1.5 * 2^23 shift on the FMA pipe, not a conversion instruction.
__device__ __forceinline__ uint32_t log_digit(float y, float& bf) {
  const float v = fminf(fmaxf(-32.f * y, 0.f), (float)(kLogBins - 1));
  const float t = v + 12582912.f;
  bf = t - 12582912.f;
  return (uint32_t)(kLogBins - 1) - (__float_as_uint(t) - 0x4B400000u);
}
__device__ __forceinline__ uint32_t log_digit(float y) {
  float bf;
  return log_digit(y, bf);
}
// The term 2^y relative to its bin's centre 2^(-b/32), in units of 2^-10:
// between about 1013 and 1035 (0 for the tiny terms of the last bin).
__device__ __forceinline__ uint32_t rel_mass(float y, float bf) {
  const float r = ex2_approx(fmaf(bf, 0.03125f, y));
  return __float_as_uint(fmaf(r, 1024.f, 12582912.f)) - 0x4B400000u;
}
// A running sum as a float pair (each addition's rounding error carried in
// lo), read out in fp64.
struct Acc {
  float hi = 0.f, lo = 0.f;
  __device__ __forceinline__ void add(float v) {
    const float sm = hi + v;
    const float bb = sm - hi;
    lo += (hi - (sm - bb)) + (v - bb);
    hi = sm;
  }
  __device__ __forceinline__ double get() const { return (double)hi + (double)lo; }
};
// Block sum of per-thread fp64 values in a fixed order (warps by xor tree,
// then warp totals in index order); every thread gets the result.
__device__ double block_sum(CutSmem& sh, double v, int lane, int warp) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFullMask, v, o);
  __syncthreads();
  if (lane == 0) sh.tsum[warp] = v;
  __syncthreads();
  double t = 0.0;
  for (int w = 0; w < kThr / 32; ++w) t += sh.tsum[w];
  __syncthreads();
  return t;
}
// The term 2^y in fixed point, units of 2^-42.
__device__ __forceinline__ unsigned long long fixed_mass(float y) {
  return __float2ull_rn(ex2_approx(y) * kFix);
}

// Calls f(x, valid) for every logit of the row; every lane of the CTA makes
// the same number of calls (valid = false past the end), so f may use
// warp-wide collectives.  Rows whose byte length is a multiple of 16 are read
// in 16-byte vectors.
template <int TT, typename F>
__device__ __forceinline__ void visit_row(const unsigned char* row, int V, F&& f) {
  constexpr int ES = TT ? 2 : 4;
  constexpr int VEC = 16 / ES;
  if (((size_t)V * ES) % 16 == 0) {
    // kLoads vectors per thread in flight before any is processed
    constexpr int kLoads = 4;
    const int nvec = V / VEC;
    for (int base = 0; base < nvec; base += kThr * kLoads) {
      uint4 w[kLoads];
      bool ok[kLoads];
#pragma unroll
      for (int u = 0; u < kLoads; ++u) {
        const int i = base + u * kThr + (int)threadIdx.x;
        ok[u] = i < nvec;
        w[u] = ok[u] ? *reinterpret_cast<const uint4*>(row + (size_t)i * 16) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < kLoads; ++u) {
        const uint32_t ws[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (TT) {
            f(bf16_lo(ws[q]), ok[u]);
            f(bf16_hi(ws[q]), ok[u]);
          } else {
            f(__uint_as_float(ws[q]), ok[u]);
          }
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

// Result of a bin scan (masses in the histogram's units, summed in fp64).
struct ScanOut {
  uint32_t digit;
  uint32_t above_cnt;  // elements in the bins above the chosen one (plus above_c0)
  double above_mass;   // their mass
  double bin_mass;     // mass of the chosen bin
  uint32_t bin_cnt;    // elements of the chosen bin
  double total;        // mass of every bin
};

// Warp 0: over NB bins with counts cnt and masses mass, the bin where the
// running sum from the top (bin NB - 1 down), added to what lies above
// (above_c0 / above_m0), first reaches the target: a count of k (BY_MASS
// false) or a mass (BY_MASS true; frac * total of these bins when
// from_total, else need_mass).  If rounding keeps the sum below the target,
// the lowest non-empty bin is taken (everything is kept).  Lane l owns bins
// [NB/32 * l, NB/32 * (l + 1)); the bins are read from shared memory twice
// rather than held in registers.
template <int NB, bool BY_MASS, typename M>
__device__ ScanOut scan_bins(const uint32_t* cnt, const M* mass, int lane, uint32_t above_c0,
                             double above_m0, uint32_t k, double need_mass, bool from_total,
                             double frac) {
  constexpr int PL = NB / 32;  // bins per lane
  const int base = PL * lane;
  uint32_t csum = 0;
  double msum = 0.0;
  for (int q = 0; q < PL; ++q) {
    csum += cnt[base + q];
    msum += (double)mass[base + q];
  }
  // sums over the lanes above (higher bins)
  uint32_t cs = csum;
  double mss = msum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_down_sync(kFullMask, cs, o);
    const double u = __shfl_down_sync(kFullMask, mss, o);
    if (lane + o < 32) {
      cs += t;
      mss += u;
    }
  }
  const uint32_t cab = cs - csum;
  const double mab = mss - msum;
  const double total = __shfl_sync(kFullMask, mss, 0);
  const double need = from_total ? frac * total : need_mass;
  int found = -1;
  uint32_t rc = cab, fc = 0, fbc = 0;
  double rm = mab, fm = 0.0, fbm = 0.0;
  for (int q = PL - 1; q >= 0; --q) {
    const uint32_t c = cnt[base + q];
    const double m = (double)mass[base + q];
    const bool hit = BY_MASS ? above_m0 + rm + m >= need : above_c0 + rc + c >= k;
    if (found < 0 && hit) {
      found = q;
      fc = rc;
      fm = rm;
      fbc = c;
      fbm = m;
    }
    rc += c;
    rm += m;
  }
  const unsigned hitmask = __ballot_sync(kFullMask, found >= 0);
  int src;
  if (hitmask) {
    src = 31 - __clz(hitmask);
  } else {  // the lowest non-empty bin
    found = -1;
    rc = cab;
    rm = mab;
    for (int q = PL - 1; q >= 0; --q) {
      const uint32_t c = cnt[base + q];
      const double m = (double)mass[base + q];
      if (c > 0) {
        found = q;
        fc = rc;
        fm = rm;
        fbc = c;
        fbm = m;
      }
      rc += c;
      rm += m;
    }
    const unsigned ne = __ballot_sync(kFullMask, found >= 0);
    src = ne ? __ffs(ne) - 1 : 0;
    if (!ne && lane == 0) {
      found = 0;
      fc = cab;
      fm = mab;
    }
  }
  ScanOut o;
  o.digit = (uint32_t)__shfl_sync(kFullMask, base + found, src);
  o.above_cnt = __shfl_sync(kFullMask, above_c0 + fc, src);
  o.above_mass = __shfl_sync(kFullMask, above_m0 + fm, src);
  o.bin_mass = __shfl_sync(kFullMask, fbm, src);
  o.bin_cnt = __shfl_sync(kFullMask, fbc, src);
  o.total = total;
  return o;
}

__device__ __forceinline__ float max_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

// The exact cut by radix levels over the keys, streaming the row once per
// level (used when the boundary bins hold more logits than the buffer).
template <int TT>
__device__ uint32_t radix_cut(CutSmem& sh, const unsigned char* rp, int V, float cT, float Rf,
                              bool use_k, bool use_p, int32_t k, float tp, int lane, int warp) {
  constexpr int NLEV = TT ? 2 : 4;
  uint32_t min_key = 0, key_k = 0, key_p = 0;
  double zk = 0.0;  // mass of the keys >= tau_k, units 2^-42
  for (int pass = 0; pass < 2; ++pass) {
    if ((pass == 0 && !use_k) || (pass == 1 && !use_p)) continue;
    uint32_t prefix = 0, above_c = 0;
    double above_m = 0.0, bin_m = 0.0;
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
        const unsigned long long fx = in ? fixed_mass(fmaf(x, cT, -Rf)) : 0ull;
        hist_add(sh, in, (u >> shift) & 0xffu, fx, lane);
      });
      __syncthreads();
      if (warp == 0) {
        const ScanOut o = pass == 0
            ? scan_bins<kBins, false>(sh.cnt, sh.mass, lane, above_c, above_m, (uint32_t)k, 0.0,
                                      false, 0.0)
            : scan_bins<kBins, true>(sh.cnt, sh.mass, lane, above_c, above_m, 0u, (double)tp * zk,
                                     !use_k && lev == 0, (double)tp);
        if (lane == 0) {
          sh.key = o.digit;
          sh.nrange = o.above_cnt;
          sh.dscr[0] = o.above_mass;
          sh.dscr[1] = o.bin_mass;
          sh.dscr[2] = o.total;
        }
      }
      __syncthreads();
      prefix |= sh.key << shift;
      above_c = sh.nrange;
      above_m = sh.dscr[0];
      bin_m = sh.dscr[1];
      if (pass == 1 && !use_k && lev == 0) zk = sh.dscr[2];
      __syncthreads();
    }
    // bf16 keys: the low 16 bits follow from the sign
    if (TT) prefix |= (prefix & 0x80000000u) ? 0u : 0xffffu;
    if (pass == 0) {
      key_k = prefix;
      min_key = prefix;
      zk = above_m + bin_m;
    } else {
      key_p = prefix;
    }
  }
  return key_k > key_p ? key_k : key_p;
}

// Sorts the first n (<= kCap) entries of the buffer by key, descending
// (bitonic network over the next power of two, at most kCap; padding keys are
// 0, below every real key).
__device__ void sort_buffer(CutSmem& sh, uint32_t n) {
  static_assert((kCap & (kCap - 1)) == 0, "the sort pads to a power of two");
  uint32_t np = 1;
  while (np < n) np <<= 1;
  for (uint32_t i = n + threadIdx.x; i < np; i += kThr) {
    sh.bkey[i] = 0u;
    sh.bmass[i] = 0ull;
  }
  __syncthreads();
  for (uint32_t size = 2; size <= np; size <<= 1) {
    for (uint32_t stride = size >> 1; stride > 0; stride >>= 1) {
      for (uint32_t i = threadIdx.x; i < np; i += kThr) {
        const uint32_t j = i ^ stride;
        if (j > i) {
          const bool desc = (i & size) == 0;
          const uint32_t a = sh.bkey[i], b = sh.bkey[j];
          if (desc ? a < b : a > b) {
            sh.bkey[i] = b;
            sh.bkey[j] = a;
            const float t = sh.bmass[i];
            sh.bmass[i] = sh.bmass[j];
            sh.bmass[j] = t;
          }
        }
      }
      __syncthreads();
    }
  }
}

// tau of a bf16 row left to the general path by the histogram kernel (a NaN
// payload no other outcome writes)
constexpr uint32_t kRetryBits = 0x7fc0a5a5u;

// The cut of one row by the general path: the row maximum, log-scale bins,
// the boundary bins collected and sorted, with radix selection behind them.
template <int TT>
__device__ void cut_row(CutSmem& sh, const unsigned char* target, int64_t row, int32_t R,
                        int32_t V, const float* temp, const int32_t* top_k, const float* top_p,
                        float* tau) {
  constexpr int ES = TT ? 2 : 4;
  const float INF = __int_as_float(0x7f800000);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
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
  // 1. the row maximum (NaN-propagating)
  float m = -INF;
  visit_row<TT>(rp, V, [&](float x, bool ok) {
    if (ok) m = max_nan(m, x);
  });
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max_nan(m, __shfl_xor_sync(kFullMask, m, o));
  if (lane == 0) sh.red[warp] = m;
  for (int i = threadIdx.x; i < kLogBins; i += kThr) {
    sh.lcnt[i] = 0;
    sh.lmassr[i] = 0;
  }
  __syncthreads();
  m = sh.red[0];
  for (int w = 1; w < kThr / 32; ++w) m = max_nan(m, sh.red[w]);
  if (m != m || m == INF || m == -INF) {  // the verifier refuses this row
    if (threadIdx.x == 0) tau[row] = -INF;
    return;
  }
  const float cT = (float)(1.4426950408889634 / (double)T);
  const float Rf = ceilf(m * cT);
  // 2. counts (exact) and masses (top-p only) of the log-scale bins; with
  // top-p and no top-k, also the row's total as a float-pair sum
  Acc s_all;
  visit_row<TT>(rp, V, [&](float x, bool ok) {
    if (!ok) return;
    const float y = fmaf(x, cT, -Rf);
    float bf;
    const uint32_t d = log_digit(y, bf);
    atomicAdd(&sh.lcnt[d], 1u);
    if (use_p) {
      atomicAdd(&sh.lmassr[d], rel_mass(y, bf));
      if (!use_k) s_all.add(ex2_approx(y));
    }
  });
  __syncthreads();
  for (int d = threadIdx.x; d < kLogBins; d += kThr)
    sh.lmass[d] = (float)sh.lmassr[d] * exp2f(-(float)(kLogBins - 1 - d) * 0.03125f - 10.f);
  __syncthreads();
  // 3. warp 0: the bins to collect, [dlo, dhi].  Top-k's bin dk is exact (from
  // the counts).  Top-p's crossing is located with the fp32 masses, the range
  // widened so that the exact crossing lies inside it barring a rounding
  // corner, which step 5 detects.
  if (warp == 0) {
    uint32_t dlo, dhi, dk = 0, above_k = 0;
    if (use_k) {
      const ScanOut o = scan_bins<kLogBins, false>(sh.lcnt, sh.lmass, lane, 0u, 0.0, (uint32_t)k,
                                                   0.0, false, 0.0);
      dk = o.digit;
      above_k = o.above_cnt;
      dlo = dhi = dk;
      if (use_p) {
        // top_p * Z_k is at least top_p * (the mass above bin dk): its
        // crossing is at or below the crossing of a little less than that
        const ScanOut a = scan_bins<kLogBins, true>(sh.lcnt, sh.lmass, lane, 0u, 0.0, 0u,
                                                    (double)tp * o.above_mass * (1.0 - 1e-4), false,
                                                    0.0);
        uint32_t d1 = a.digit;
        uint32_t hi_ne = 0;  // a target of 0 is met at the top: the highest non-empty bin
#pragma unroll
        for (int q = 0; q < kLogBins / 32; ++q)
          if (sh.lcnt[(kLogBins / 32) * lane + q] > 0) hi_ne = (kLogBins / 32) * lane + q;
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) hi_ne = max(hi_ne, __shfl_xor_sync(kFullMask, hi_ne, o2));
        if (d1 > hi_ne) d1 = hi_ne;
        dhi = d1 > dk ? d1 : dk;
      }
    } else {
      const ScanOut o = scan_bins<kLogBins, true>(sh.lcnt, sh.lmass, lane, 0u, 0.0, 0u, 0.0, true,
                                                  (double)tp);
      dlo = o.digit > 0 ? o.digit - 1 : 0;
      dhi = o.digit < kLogBins - 1 ? o.digit + 1 : kLogBins - 1;
    }
    uint32_t nr = 0, nab = 0;
#pragma unroll
    for (int q = 0; q < kLogBins / 32; ++q) {
      const uint32_t d = (kLogBins / 32) * lane + q;
      if (d >= dlo && d <= dhi) nr += sh.lcnt[d];
      if (d > dk && d <= dhi) nab += sh.lcnt[d];
    }
    nr = __reduce_add_sync(kFullMask, nr);
    nab = __reduce_add_sync(kFullMask, nab);
    if (lane == 0) {
      sh.dlo = dlo;
      sh.dhi = dhi;
      sh.nrange = nr;
      sh.above_in_range = nab;
      sh.nbuf = 0;
      sh.key = dk;
      sh.idx = above_k;
    }
  }
  __syncthreads();
  const uint32_t dlo = sh.dlo, dhi = sh.dhi, nrange = sh.nrange;
  const uint32_t dk = sh.key, above_k = sh.idx, nab = sh.above_in_range;
  bool fallback = nrange > (uint32_t)kCap;
  uint32_t key_k = 0, key_p = 0;
  if (!fallback) {
    __syncthreads();
    // 4. the logits of bins [dlo, dhi] into the buffer; float-pair sums of the
    // terms above dhi (top-p) and above dk (top-k); logits below the range
    // need nothing
    Acc s_hi, s_k;
    visit_row<TT>(rp, V, [&](float x, bool ok) {
      if (!ok) return;
      const float y = fmaf(x, cT, -Rf);
      const uint32_t d = log_digit(y);
      if (d < dlo) return;
      const float e = ex2_approx(y);
      if (use_k && d > dk) s_k.add(e);
      if (use_p && d > dhi) s_hi.add(e);
      if (d <= dhi) {
        const uint32_t pos = atomicAdd(&sh.nbuf, 1u);
        if (pos < (uint32_t)kCap) {
          sh.bkey[pos] = order_key(x);
          sh.bmass[pos] = e;
        }
      }
    });
    const double base_mass = use_p ? block_sum(sh, s_hi.get(), lane, warp) : 0.0;
    const double above_mk = use_k ? block_sum(sh, s_k.get(), lane, warp) : 0.0;
    const double total = use_k ? 0.0 : block_sum(sh, s_all.get(), lane, warp);
    const uint32_t n = min(sh.nbuf, (uint32_t)kCap);
    __syncthreads();
    sort_buffer(sh, n);
    // 5. the cuts, from the sorted buffer
    double zk = total;
    if (use_k) {
      key_k = sh.bkey[nab + (uint32_t)k - above_k - 1];
      // Z_k: the mass above bin dk and that of bin dk's logits >= tau_k
      double part = 0.0;
      for (uint32_t i = nab + threadIdx.x; i < n; i += kThr)
        if (sh.bkey[i] >= key_k) part += (double)sh.bmass[i];
      zk = above_mk + block_sum(sh, part, lane, warp);
    }
    if (use_p) {
      const double need = (double)tp * zk - base_mass;
      // running mass over the sorted buffer (logits >= tau_k): per-thread
      // chunks, their exclusive prefix by warp 0, then each chunk walked
      const uint32_t chunk = (n + kThr - 1) / kThr;
      const uint32_t i0 = min(n, threadIdx.x * chunk), i1 = min(n, i0 + chunk);
      double own = 0.0;
      for (uint32_t i = i0; i < i1; ++i)
        if (sh.bkey[i] >= key_k) own += (double)sh.bmass[i];
      sh.tsum[threadIdx.x] = own;
      if (threadIdx.x == 0) sh.idx = 0xffffffffu;
      __syncthreads();
      if (warp == 0) {
        constexpr int PT = kThr / 32;
        double v[PT], t = 0.0;
#pragma unroll
        for (int q = 0; q < PT; ++q) {
          v[q] = sh.tsum[PT * lane + q];
          t += v[q];
        }
        double incl = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const double u = __shfl_up_sync(kFullMask, incl, o);
          if (lane >= o) incl += u;
        }
        double run = incl - t;
#pragma unroll
        for (int q = 0; q < PT; ++q) {
          sh.tsum[PT * lane + q] = run;
          run += v[q];
        }
      }
      __syncthreads();
      double run = sh.tsum[threadIdx.x];
      for (uint32_t i = i0; i < i1; ++i) {
        if (sh.bkey[i] < key_k) continue;
        run += (double)sh.bmass[i];
        if (run >= need) {
          atomicMin(&sh.idx, i);
          break;
        }
      }
      __syncthreads();
      const uint32_t ix = sh.idx;
      if (!(need > 0.0)) {
        fallback = true;  // the crossing lies above the collected bins
      } else if (ix != 0xffffffffu) {
        key_p = sh.bkey[ix];
      } else if (use_k || dlo == 0) {
        // no crossing inside: every logit >= tau_k (or the whole row) is kept
        key_p = 0;
      } else {
        fallback = true;  // the crossing lies below the collected bins
      }
    }
  }
  if (fallback) {  // uniform over the CTA
    __syncthreads();
    const uint32_t key = radix_cut<TT>(sh, rp, V, cT, Rf, use_k, use_p, k, tp, lane, warp);
    if (threadIdx.x == 0) tau[row] = key_value(key);
    return;
  }
  // key 0: nothing cut (top-p keeps the whole row)
  const uint32_t key = key_k > key_p ? key_k : key_p;
  if (threadIdx.x == 0) tau[row] = key ? key_value(key) : -INF;
}

// Rows blockIdx.x, blockIdx.x + gridDim.x, ... by the general path; with
// only_marked, just the rows whose tau holds kRetryBits.
template <int TT>
__global__ void __launch_bounds__(kThr, 4) cut_kernel(const unsigned char* target, int64_t rows,
                                                   int32_t R, int32_t V, const float* temp,
                                                   const int32_t* top_k, const float* top_p,
                                                   float* tau, int only_marked) {
  extern __shared__ __align__(16) unsigned char cut_dsm[];
  CutSmem& sh = *reinterpret_cast<CutSmem*>(cut_dsm);
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    if (only_marked && __float_as_uint(tau[row]) != kRetryBits) continue;
    __syncthreads();  // the previous row is done with the shared memory
    cut_row<TT>(sh, target, row, R, V, temp, top_k, top_p, tau);
  }
}

// ---- bf16 rows: an exact count per bit pattern ------------------------------
//
// A bf16 logit is one of 65,536 bit patterns, so a count per pattern describes
// the row exactly: the k-th largest value and every mass sum follow from the
// counts, with no sort and no exponential per logit.  Counts are the 16-bit
// halves of 32-bit shared-memory words (pattern p in word p >> 1, half p & 1;
// 128 KB).  A row holding more than 65,535 copies of one value wraps a half;
// the total count shows it, and such a row is marked for the general path (a
// second launch that cuts only the marked rows).  Each row is streamed once,
// one shared atomic per logit, with the row maximum (as a value-order key)
// tracked on the way.  A mass is computed once per non-empty pattern,
// count x 2^((v - vmax) log2(e) / T) in fixed point (units of 2^-42), so
// every prefix sum is exact and independent of the order of the additions,
// and the top-p crossing is decided exactly.
//
// The patterns fall into 1024 chunks of 64 (32 words), chunk t owned by
// thread t.  Chunks below 512 hold positive values (larger with the index),
// the others negative ones (smaller with the index), so in descending order
// of value they come as 511, 510, ..., 0, 512, ..., 1023 (+0 and -0, patterns
// 0 and 0x8000, meet at the seam).  After the pass each thread sums its
// chunk's counts and masses (lane l starting at word l of its chunk, so a
// warp's reads hit distinct banks), one block scan in that order locates the
// chunks where the running count reaches k and the running mass reaches
// ceil(top_p * Z_k), and a warp walks each of those chunks, one word per lane.
//
// One persistent CTA of 1024 threads per SM takes rows blockIdx.x,
// blockIdx.x + gridDim.x, ...; each row's parameters are loaded while the
// previous row is cut.

constexpr int kHT = 1024;       // threads of the histogram kernel (one per chunk)
constexpr int kHWords = 32768;  // 65,536 patterns, two counts per word
constexpr int kChunks = 1024;   // 64 patterns, 32 words each
static_assert(kChunks == kHT && kHWords == 32 * kChunks, "one chunk per thread");

struct HistScratch {
  unsigned long long cmass[kChunks];  // per-chunk masses
  uint32_t ccnt[kChunks];             // per-chunk counts
  unsigned long long wm[32];  // per-warp scan totals (masses), by rank
  uint32_t wc[32];            // per-warp scan totals (counts), by rank
  uint32_t wsp[32];           // per-warp flags
  uint32_t wmax[32];          // per-warp largest value-order keys
  unsigned long long kmrun, prun;
  uint32_t krun, kchunk, pchunk;
};

// Value order of a pattern: okey16(a) > okey16(b) iff value(a) > value(b)
// (NaN patterns aside; -0 sits just below +0).
__device__ __forceinline__ uint32_t okey16(uint32_t p) {
  return p < 0x8000u ? 0x8000u + p : 0xffffu - p;
}
// okey16 of both patterns of a word at once.
__device__ __forceinline__ uint32_t okey16x2(uint32_t w) {
  const uint32_t s2 = (w >> 15) & 0x00010001u;
  return w ^ (s2 * 0x7fffu) ^ 0x80008000u;
}
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ float pattern_value(uint32_t p) { return __uint_as_float(p << 16); }
__device__ __forceinline__ uint32_t half_count(uint32_t w, uint32_t p) {
  return (p & 1u) ? (w >> 16) : (w & 0xffffu);
}
// Exclusive prefixes, in descending order of the threads' chunks, of the
// per-thread counts c and masses m (the masses only when with_mass), with
// their totals, and the OR of the flags f.  One barrier; called by every
// thread.
struct ChunkScan {
  uint32_t c_ex, c_tot, flags;
  unsigned long long m_ex, m_tot;
};
__device__ ChunkScan chunk_scan(HistScratch& hs, uint32_t c, unsigned long long m, uint32_t f,
                                bool with_mass, int lane, int warp) {
  const bool rev = warp < kHT / 64;  // positive chunks: higher lanes come first
  uint32_t ci = c;
  unsigned long long mi = with_mass ? m : 0ull;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const bool take = rev ? lane + o < 32 : lane >= o;
    const uint32_t uc = rev ? __shfl_down_sync(kFullMask, ci, o) : __shfl_up_sync(kFullMask, ci, o);
    if (take) ci += uc;
    if (with_mass) {
      const unsigned long long um =
          rev ? __shfl_down_sync(kFullMask, mi, o) : __shfl_up_sync(kFullMask, mi, o);
      if (take) mi += um;
    }
  }
  const uint32_t wf = __reduce_or_sync(kFullMask, f);
  const int wr = rev ? kHT / 64 - 1 - warp : warp;
  if (lane == (rev ? 0 : 31)) {
    hs.wc[wr] = ci;
    hs.wm[wr] = mi;
    hs.wsp[wr] = wf;
  }
  __syncthreads();
  ChunkScan o;
  o.flags = __reduce_or_sync(kFullMask, hs.wsp[lane]);
  const uint32_t tc = hs.wc[lane];
  uint32_t tci = tc;
#pragma unroll
  for (int q = 1; q < 32; q <<= 1) {
    const uint32_t u = __shfl_up_sync(kFullMask, tci, q);
    if (lane >= q) tci += u;
  }
  o.c_ex = __shfl_sync(kFullMask, tci - tc, wr) + ci - c;
  o.c_tot = __shfl_sync(kFullMask, tci, 31);
  o.m_ex = o.m_tot = 0;
  if (with_mass) {
    const unsigned long long tm = hs.wm[lane];
    unsigned long long tmi = tm;
#pragma unroll
    for (int q = 1; q < 32; q <<= 1) {
      const unsigned long long u = __shfl_up_sync(kFullMask, tmi, q);
      if (lane >= q) tmi += u;
    }
    o.m_ex = __shfl_sync(kFullMask, tmi - tm, wr) + mi - m;
    o.m_tot = __shfl_sync(kFullMask, tmi, 31);
  }
  return o;
}

// Walks chunk c in descending order of value, one word per lane, from `run`
// (the weight of everything above the chunk) and returns the first pattern at
// which the running weight reaches `target` (the chunk's last non-empty one
// if it never does).  weight(c, p): the weight of the c logits of pattern p.
template <typename U, typename Wt>
__device__ uint32_t chunk_step(const uint32_t* hist, uint32_t c, int lane, U run, U target,
                               Wt&& weight) {
  const bool pos = c < kChunks / 2;
  const uint32_t word = 32 * c + (pos ? 31 - lane : lane);
  const uint32_t w = hist[word];
  const uint32_t pf = pos ? 2 * word + 1 : 2 * word;  // the larger value of the two
  const uint32_t ps = pf ^ 1u;
  const U a = weight(half_count(w, pf), pf);
  const U b = weight(half_count(w, ps), ps);
  U inc = a + b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const U u = __shfl_up_sync(kFullMask, inc, o);
    if (lane >= o) inc += u;
  }
  const U before = run + inc - a - b;
  unsigned hit = __ballot_sync(kFullMask, before + a + b >= target);
  uint32_t res = before + a >= target ? pf : ps;
  if (!hit) {  // not reached: the last pattern with weight
    hit = __ballot_sync(kFullMask, a + b > 0);
    res = b > 0 ? ps : pf;
    return hit ? __shfl_sync(kFullMask, res, 31 - __clz(hit)) : pf;
  }
  return __shfl_sync(kFullMask, res, __ffs(hit) - 1);
}

// ceil(tp * Z) for a float tp in (0, 1) and Z < 2^63, exactly.
__device__ __forceinline__ unsigned long long mul_ceil(unsigned long long Z, float tp) {
  const uint32_t bits = __float_as_uint(tp);
  uint32_t e = bits >> 23;
  unsigned long long m = bits & 0x7fffffu;
  if (e) m |= 0x800000u;
  else e = 1;
  const int s = 150 - (int)e;  // tp = m 2^-s, s >= 24
  const unsigned long long lo = Z * m, hi = __umul64hi(Z, m);
  unsigned long long q;
  bool rem;
  if (s < 64) {
    q = (lo >> s) | (hi << (64 - s));
    rem = (lo & ((1ull << s) - 1)) != 0;
  } else if (s < 128) {
    const int r = s - 64;
    q = r ? hi >> r : hi;
    rem = lo != 0 || (r && (hi & ((1ull << r) - 1)) != 0);
  } else {
    q = 0;
    rem = lo != 0 || hi != 0;
  }
  return q + (rem ? 1ull : 0ull);
}

// floor(t 2^42) for t in [0, 1], from the float's fields (no conversion
// instruction).
__device__ __forceinline__ unsigned long long fixed42(float t) {
  const uint32_t bits = __float_as_uint(t);
  const int e = (int)(bits >> 23);
  const uint32_t m = (bits & 0x7fffffu) | 0x800000u;
  if (e >= 108) return (unsigned long long)m << ((e - 108) & 63);
  return e > 84 ? (unsigned long long)(m >> (108 - e)) : 0ull;
}

// Sum over the warp of values below 2^63 (three 21-bit parts through
// redux.sync).
__device__ __forceinline__ unsigned long long warp_sum63(unsigned long long v) {
  const uint32_t p0 = __reduce_add_sync(kFullMask, (uint32_t)(v & 0x1fffffu));
  const uint32_t p1 = __reduce_add_sync(kFullMask, (uint32_t)((v >> 21) & 0x1fffffu));
  const uint32_t p2 = __reduce_add_sync(kFullMask, (uint32_t)(v >> 42));
  return (unsigned long long)p0 + ((unsigned long long)p1 << 21) + ((unsigned long long)p2 << 42);
}

// Adds the two bf16 patterns of word w to the histogram.
__device__ __forceinline__ void count_pair(uint32_t* hist, uint32_t w) {
  atomicAdd(&hist[(w >> 1) & 0x7fffu], (w & 1u) * 0xffffu + 1u);
  atomicAdd(&hist[w >> 17], ((w >> 16) & 1u) * 0xffffu + 1u);
}

__global__ void __launch_bounds__(kHT, 1)
    cut_hist_kernel(const unsigned char* target, int64_t rows, int32_t R, int32_t V,
                    const float* temp, const int32_t* top_k, const float* top_p, float* tau) {
  extern __shared__ __align__(16) unsigned char hist_dsm[];
  uint32_t* hist = reinterpret_cast<uint32_t*>(hist_dsm);
  HistScratch& hs = *reinterpret_cast<HistScratch*>(hist_dsm + (size_t)kHWords * 4);
  const float INF = __int_as_float(0x7f800000);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const size_t row_bytes = (size_t)V * 2;
  float nT = 0.f, ntp = 0.f;
  int32_t nk = 0;
  if ((int64_t)blockIdx.x < rows) {
    const int64_t b = blockIdx.x / R;
    nT = temp[b];
    nk = top_k[b];
    ntp = top_p[b];
  }
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    const float T = nT, tp = ntp;
    const int32_t k = nk;
    if (row + gridDim.x < rows) {  // the next row's parameters, used next iteration
      const int64_t b = (row + gridDim.x) / R;
      nT = temp[b];
      nk = top_k[b];
      ntp = top_p[b];
    }
    if (!(T > 0.f) || !(T < INF) || !(tp > 0.f)) {
      if (tid == 0) tau[row] = __int_as_float(0x7fc00000);
      continue;
    }
    const bool use_k = k > 0 && k < V;
    const bool use_p = tp < 1.f;
    if (!use_k && !use_p) {
      if (tid == 0) tau[row] = -INF;
      continue;
    }
    const unsigned char* rp = target + (size_t)row * row_bytes;
    __syncthreads();  // the previous row's readers are done
    for (int i = tid; i < kHWords / 4; i += kHT)
      reinterpret_cast<uint4*>(hist)[i] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    // 1. one pass over the row: a count per bit pattern, and the largest
    // value-order key
    uint32_t kmax2 = 0;
    if ((row_bytes & 15) == 0) {
      const uint4* rv = reinterpret_cast<const uint4*>(rp);
      const int nvec = V >> 3;
      constexpr int kLoads = 4;
      for (int base = 0; base < nvec; base += kHT * kLoads) {
        uint4 w[kLoads];
#pragma unroll
        for (int u = 0; u < kLoads; ++u) {
          const int i = base + u * kHT + tid;
          if (i < nvec) w[u] = __ldcs(rv + i);
        }
#pragma unroll
        for (int u = 0; u < kLoads; ++u) {
          if (base + u * kHT + tid < nvec) {
            count_pair(hist, w[u].x);
            count_pair(hist, w[u].y);
            count_pair(hist, w[u].z);
            count_pair(hist, w[u].w);
            kmax2 = max_u16x2(kmax2, max_u16x2(max_u16x2(okey16x2(w[u].x), okey16x2(w[u].y)),
                                               max_u16x2(okey16x2(w[u].z), okey16x2(w[u].w))));
          }
        }
      }
    } else {
      const uint16_t* rs = reinterpret_cast<const uint16_t*>(rp);
      for (int i = tid; i < V; i += kHT) {
        const uint32_t p = rs[i];
        atomicAdd(&hist[p >> 1], (p & 1u) * 0xffffu + 1u);
        kmax2 = max(kmax2, okey16(p));
      }
    }
    {
      const uint32_t km = __reduce_max_sync(kFullMask, max(kmax2 & 0xffffu, kmax2 >> 16));
      if (lane == 0) hs.wmax[warp] = km;
    }
    __syncthreads();
    const uint32_t kmax = __reduce_max_sync(kFullMask, hs.wmax[lane]);
    const float vmax = pattern_value(kmax >= 0x8000u ? kmax - 0x8000u : 0xffffu - kmax);
    const float cT = 1.44269504088896341f / T;
    // a pattern's mass, count x 2^((v - vmax) log2(e) / T), units of 2^-42
    const auto mass = [=](uint32_t c, uint32_t p) -> unsigned long long {
      return (unsigned long long)c * fixed42(ex2_approx((pattern_value(p) - vmax) * cT));
    };
    // 2. the count and (top-p) the mass of every chunk.  Four lanes share a
    // chunk, 8 words each, so a warp covers 8 chunks per round and the dense
    // chunks of a row (consecutive) spread over several warps; lane l starts
    // at word (l / 4) of its quarter, so a warp's 32 reads hit 32 banks.
    for (int rd = 0; rd < kChunks / kHT * 4; ++rd) {
      const int c = 8 * (rd * (kHT / 32) + warp) + (lane >> 2);
      const int w0 = 32 * c + 8 * (lane & 3);
      uint32_t cc = 0;
      unsigned long long cm = 0;
#pragma unroll
      for (int i = 0; i < 8; i += 4) {
        uint32_t wd[4], w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          wd[u] = w0 + ((i + u + (lane >> 2)) & 7);
          w[u] = hist[wd[u]];
          cc += (w[u] & 0xffffu) + (w[u] >> 16);
        }
        if (use_p && (w[0] | w[1] | w[2] | w[3])) {
#pragma unroll
          for (int u = 0; u < 4; ++u)
            cm += mass(w[u] & 0xffffu, 2 * wd[u]) + mass(w[u] >> 16, 2 * wd[u] + 1);
        }
      }
#pragma unroll
      for (int o = 1; o < 4; o <<= 1) {
        cc += __shfl_xor_sync(kFullMask, cc, o);
        if (use_p) cm += __shfl_xor_sync(kFullMask, cm, o);
      }
      if ((lane & 3) == 0) {
        hs.ccnt[c] = cc;
        hs.cmass[c] = cm;
      }
    }
    __syncthreads();
    // thread t: chunk t.  Chunks 510, 511 and 1023 hold only +inf and NaN
    // patterns, chunk 1022 -inf (pattern 0xff80, the low half of its first
    // word) and NaNs.
    const uint32_t cnt = hs.ccnt[tid];
    const unsigned long long mine = use_p ? hs.cmass[tid] : 0ull;
    uint32_t special = 0;
    if (tid == 510 || tid == 511 || tid == 1023) special = cnt != 0;
    else if (tid == 1022) special = cnt != (hist[0x7fc0] & 0xffffu);
    const ChunkScan sc = chunk_scan(hs, cnt, mine, special, use_p, lane, warp);
    if (sc.c_tot != (uint32_t)V) {
      // a count wrapped: the row goes to the general path (a second launch)
      if (tid == 0) tau[row] = __uint_as_float(kRetryBits);
      continue;
    }
    // the verifier refuses rows with a NaN or +inf, and rows of -inf only
    if (sc.flags || kmax >= 0xff80u || kmax <= okey16(0xff80u)) {
      if (tid == 0) tau[row] = -INF;
      continue;
    }
    // 3. the crossing chunks: top-k's where the count from the top reaches k;
    // top-p's where the mass from the top reaches ceil(top_p * Z_k), Z_k the
    // mass of the patterns >= tau_k
    float cut = -INF;
    unsigned long long need = 0;
    if (use_k) {
      if (sc.c_ex < (uint32_t)k && sc.c_ex + cnt >= (uint32_t)k) {
        hs.kchunk = tid;
        hs.krun = sc.c_ex;
        hs.kmrun = sc.m_ex;
      }
    } else {
      need = mul_ceil(sc.m_tot, tp);
      if (sc.m_ex < need && sc.m_ex + mine >= need) {
        hs.pchunk = tid;
        hs.prun = sc.m_ex;
      }
    }
    __syncthreads();
    if (use_k) {
      const uint32_t kc = hs.kchunk;
      cut = pattern_value(chunk_step<uint32_t>(hist, kc, lane, hs.krun, (uint32_t)k,
                                               [](uint32_t c, uint32_t) { return c; }));
      if (use_p) {
        // Z_k: the mass above chunk kc and that of kc's patterns >= tau_k
        const uint32_t word = 32 * kc + lane;
        const uint32_t w = hist[word];
        unsigned long long part = 0;
        if (pattern_value(2 * word) >= cut) part += mass(w & 0xffffu, 2 * word);
        if (pattern_value(2 * word + 1) >= cut) part += mass(w >> 16, 2 * word + 1);
        // tau_k = +0 keeps the -0 logits too (pattern 0x8000, chunk 512)
        if (kc == 0 && lane == 0) part += mass(hist[0x4000] & 0xffffu, 0x8000u);
        need = mul_ceil(hs.kmrun + warp_sum63(part), tp);
        if (sc.m_ex < need && sc.m_ex + mine >= need) {
          hs.pchunk = tid;
          hs.prun = sc.m_ex;
        }
        __syncthreads();
      }
    }
    // 4. top-p: the pattern of its crossing chunk where the mass reaches need
    // (at or above tau_k: the inclusive mass at tau_k is Z_k)
    if (use_p) cut = pattern_value(chunk_step<unsigned long long>(hist, hs.pchunk, lane, hs.prun,
                                                                  need, mass));
    if (tid == 0) tau[row] = cut;
  }
}

}  // namespace

int launch_sampling_cut(const void* target, int32_t dtype, int32_t B, int32_t R, int32_t V,
                        const float* temp, const int32_t* top_k, const float* top_p, float* tau,
                        cudaStream_t stream) {
  const int64_t rows = (int64_t)B * R;
  const auto* t = static_cast<const unsigned char*>(target);
  // the kernels' shared-memory opt-in and the SM count, once per device (no
  // runtime call besides the launch afterwards, so launches can be captured
  // in graphs)
  constexpr int kMaxDev = 64;
  static bool attr_done[kMaxDev] = {false};
  static int sm_count[kMaxDev] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return SAMSPEC_ECUDA;
  const int smem = (int)sizeof(CutSmem);
  const int hsmem = kHWords * 4 + (int)sizeof(HistScratch);
  if (!attr_done[dev]) {
    if (cudaFuncSetAttribute(cut_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
            cudaSuccess ||
        cudaFuncSetAttribute(cut_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
            cudaSuccess ||
        cudaFuncSetAttribute(cut_hist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             hsmem) != cudaSuccess ||
        cudaDeviceGetAttribute(&sm_count[dev], cudaDevAttrMultiProcessorCount, dev) !=
            cudaSuccess ||
        sm_count[dev] < 1)
      return SAMSPEC_ECUDA;
    attr_done[dev] = true;
  }
  if (dtype == SAMSPEC_F32) {
    cut_kernel<0><<<(unsigned)rows, kThr, smem, stream>>>(t, rows, R, V, temp, top_k, top_p, tau,
                                                          0);
  } else {
    const int64_t grid = rows < sm_count[dev] ? rows : sm_count[dev];
    cut_hist_kernel<<<(unsigned)grid, kHT, hsmem, stream>>>(t, rows, R, V, temp, top_k, top_p,
                                                            tau);
    if (cudaGetLastError() != cudaSuccess) return SAMSPEC_ECUDA;
    const int64_t g2 = rows < 4 * (int64_t)sm_count[dev] ? rows : 4 * (int64_t)sm_count[dev];
    cut_kernel<1><<<(unsigned)g2, kThr, smem, stream>>>(t, rows, R, V, temp, top_k, top_p, tau, 1);
  }
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
