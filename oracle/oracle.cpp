// oracle.cpp -- plain, slow, single-threaded CPU reference for the SAM-drafting
// + lossless-verification hot path.
//
// TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes or
// calls this file.  Only the tests, the package smoke check and the benchmark's
// CPU-baseline / reference arm load it.  It shares no code, header, table or
// constant generator with the CUDA path: every step here is written out from the
// pages' description, in fp64 wherever the arithmetic is floating point.
//
// Pages followed (titles as printed; sections named as on each page):
//   [P1] "SAM投机推理：长序列强化学习训练加速利器" (CANN cann-recipes-train article)
//        §1.1 SAM 原理: endpos / endpos classes, link, next, the ABCBC example,
//        dynamic SAM (D-SAM) extended after every verified token, min_endpos,
//        draft generation by walking link edges, rejection test eps <= alpha(x).
//   [P2] nxbn.cn speculative-sampling article, §2.2 验证阶段的并行打分机制:
//        accept with probability min(1, p_target/p_draft); on rejection resample
//        from the positive part of (p_target - p_draft); K+1 distributions.
//   [P3] gogongxt.com notes "投机采样", sections 贪婪采样 / 拒绝采样 /
//        SGLang 的实现 / N-gram 的特殊情况: greedy = keep drafts equal to the
//        target argmax; softmax(logits / temperature); draft_probs = 0 for
//        model-free drafts (q is one-hot at the draft token), bonus sampling
//        then degenerates to sampling the target distribution.
//   [P4] volcengine.com SAM-Decoding article, §3 "Suffix Automaton
//        Construction" (Blumer's online construction, min_endpos per node),
//        "Drafting with Suffix Automaton", "Update of Suffix Automaton"
//        (dynamic automaton: extend first, then move the matching state).
//
// Philox4x32-10 is not on the pages; it is written from its published
// definition (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
// 1, 2, 3", SC'11): 10 rounds, multipliers 0xD2511F53 / 0xCD9E8D57, Weyl key
// increments 0x9E3779B9 / 0xBB67AE85.
//
// Readings where the pages are silent (each listed in the design notes):
//   positions are 0-based (endpos(BC) = {2,4} in ABCBC, [P1] §1.1);
//   state ids: the new state `cur` is numbered before its `clone`;
//   zero-length match -> no draft, match_len 0, min_endpos -1;
//   a draft running past the end of the text is truncated;
//   greedy ties -> lowest token id; accept iff u * q(d) <= p(d);
//   temperature applies to draft logits too; residual of mass 0 -> sample p;
//   CDF walked in ascending token id with a strict ">" test; if rounding leaves
//   the whole CDF <= t, the largest token with positive residual is taken.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <limits>
#include <map>
#include <vector>

namespace {

// ---------------------------------------------------------------------------
// Suffix automaton ([P1] §1.1, [P4] §3).  One object per sequence.
// ---------------------------------------------------------------------------
struct Sam {
  int32_t vocab = 0;
  std::vector<int32_t> len;        // length of the longest string of each state
  std::vector<int32_t> link;       // suffix link (-1 at the root)
  std::vector<int32_t> min_endpos; // smallest end position of the state's strings
  std::vector<std::map<int32_t, int32_t>> next;  // next[state][token] = state
  std::vector<int32_t> text;       // the reference string S = s_0 ... s_{n-1}
  int32_t last = 0;                // state of the whole string S
  int64_t walk_steps = 0;          // link-walk iterations over all extensions

  explicit Sam(int32_t v) : vocab(v) { new_state(0, -1, -1); }

  int32_t new_state(int32_t l, int32_t lk, int32_t me) {
    len.push_back(l);
    link.push_back(lk);
    min_endpos.push_back(me);
    next.emplace_back();
    return (int32_t)len.size() - 1;
  }

  // Append one token c at position i = |S| (Blumer et al.'s online step,
  // cited by [P4] §3; the D-SAM update of [P1] §1.1).
  void extend(int32_t c) {
    const int32_t i = (int32_t)text.size();
    // the new position i ends only the suffixes of S c; it is larger than any
    // earlier end position, so `cur` records i as its smallest end position.
    const int32_t cur = new_state(len[last] + 1, -1, i);
    int32_t p = last;
    while (p != -1 && next[p].find(c) == next[p].end()) {
      next[p][c] = cur;
      p = link[p];
      ++walk_steps;
    }
    if (p == -1) {
      link[cur] = 0;
    } else {
      const int32_t q = next[p][c];
      if (len[p] + 1 == len[q]) {
        link[cur] = q;
      } else {
        // split q: the clone keeps q's transitions, suffix link and smallest
        // end position (its strings occur wherever q's shorter strings do).
        const int32_t clone = new_state(len[p] + 1, link[q], min_endpos[q]);
        next[clone] = next[q];
        while (p != -1) {
          auto it = next[p].find(c);
          if (it == next[p].end() || it->second != q) break;
          it->second = clone;
          p = link[p];
          ++walk_steps;
        }
        link[q] = clone;
        link[cur] = clone;
      }
    }
    last = cur;
    text.push_back(c);
  }

  // Draft query ([P1] §1.1 草稿生成; [P4] "Drafting with Suffix Automaton"):
  // from the state of S walk link edges until a state has a next edge; its
  // longest string is the longest suffix of S that also ends earlier in S.
  // The draft copies the tokens that followed its first occurrence.
  void draft(int32_t K, int32_t* out, int32_t* draft_len, int32_t* match_len,
             int32_t* min_end) const {
    int32_t v = last;
    while (v != 0 && next[v].empty()) v = link[v];
    const int32_t n = (int32_t)text.size();
    *match_len = len[v];
    *min_end = min_endpos[v];
    int32_t dl = 0;
    if (v != 0) {
      const int32_t e = min_endpos[v];
      dl = n - 1 - e;
      if (dl > K) dl = K;
      for (int32_t t = 0; t < dl; ++t) out[t] = text[e + 1 + t];
    }
    for (int32_t t = dl; t < K; ++t) out[t] = -1;
    *draft_len = dl;
  }

  // Static use ([P4] "Drafting with Suffix Automaton", "Update of Suffix
  // Automaton"; [P1] §1.1 静态 SAM): this automaton holds a corpus and stays
  // fixed; a generated text is followed by a matching state (v, l): v the
  // state of the longest suffix of the generated text that occurs in the
  // corpus, l its length.  A new token c moves it along c if v has that
  // transition; otherwise shorter suffixes are tried by following links
  // (their longest string, len(link)), and with none left the match is
  // empty (root, 0).
  void match(int32_t* v_io, int32_t* l_io, int32_t c) const {
    int32_t v = *v_io, l = *l_io;
    while (v != 0 && next[v].find(c) == next[v].end()) {
      v = link[v];
      l = len[v];
    }
    auto it = next[v].find(c);
    if (it != next[v].end()) {
      v = it->second;
      l = l + 1;
    } else {
      v = 0;
      l = 0;
    }
    *v_io = v;
    *l_io = l;
  }

  // Draft from a matching state: the K corpus tokens after the first
  // occurrence (min_endpos) of the matched suffix, cut at the corpus end.
  void match_draft(int32_t v, int32_t l, int32_t K, int32_t* out, int32_t* draft_len) const {
    const int32_t n = (int32_t)text.size();
    int32_t dl = 0;
    if (v != 0 && l > 0) {
      const int32_t e = min_endpos[v];
      dl = n - 1 - e;
      if (dl > K) dl = K;
      for (int32_t t = 0; t < dl; ++t) out[t] = text[e + 1 + t];
    }
    for (int32_t t = dl; t < K; ++t) out[t] = -1;
    *draft_len = dl;
  }
};

// ---------------------------------------------------------------------------
// Philox4x32-10 and the uniform map.
// ---------------------------------------------------------------------------
void philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {  // key schedule: Weyl increments between rounds
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint64_t prod0 = (uint64_t)0xD2511F53u * (uint64_t)x0;
    const uint64_t prod1 = (uint64_t)0xCD9E8D57u * (uint64_t)x2;
    const uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
    const uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
    const uint32_t y0 = hi1 ^ x1 ^ k0;
    const uint32_t y1 = lo1;
    const uint32_t y2 = hi0 ^ x3 ^ k1;
    const uint32_t y3 = lo0;
    x0 = y0; x1 = y1; x2 = y2; x3 = y3;
  }
  out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

// U(x) = ((x >> 9) + 1/2) * 2^-23, in (0, 1); exact in binary32 and binary64.
double uniform_from_word(uint32_t x) {
  return ((double)(x >> 9) + 0.5) * (1.0 / 8388608.0);
}

// Uniforms of sequence b at draft position j: word 0 drives the accept test,
// word 1 the resample.  key = (seed lo, seed hi), counter = (j, b, step lo, step hi).
void uniforms(uint64_t seed, uint64_t step, int64_t b, int32_t j, double* u_acc,
              double* u_res) {
  const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  const uint32_t ctr[4] = {(uint32_t)j, (uint32_t)b, (uint32_t)step, (uint32_t)(step >> 32)};
  uint32_t out[4];
  philox4x32_10(ctr, key, out);
  *u_acc = uniform_from_word(out[0]);
  *u_res = uniform_from_word(out[1]);
}

// ---------------------------------------------------------------------------
// Verification ([P2] §2.2; [P3] 贪婪采样, 拒绝采样, N-gram 的特殊情况).
// ---------------------------------------------------------------------------
enum : int32_t {
  OV_OK = 0,
  OV_BADROW = 5,    // NaN, +inf (T > 0) or an all -inf row
  OV_BADDRAFT = 6,  // draft length outside [0, K] or draft token outside [0, V)
  OV_BADPARAM = 8,  // sampling parameters: T not > 0 and finite, or top_p not > 0
};

// Greedy: argmax with the lowest index on ties.  Returns false for a row the
// argmax is not defined on (a NaN, or every entry -inf).
bool argmax_row(const float* row, int32_t V, int32_t* arg, double* maxval) {
  int32_t best = -1;
  double bv = -std::numeric_limits<double>::infinity();
  for (int32_t v = 0; v < V; ++v) {
    const double x = (double)row[v];
    if (std::isnan(x)) return false;
    if (x > bv) { bv = x; best = v; }
  }
  if (best < 0) return false;
  *arg = best;
  *maxval = bv;
  return true;
}

// Temperature softmax in fp64: x_v = l_v / T, m = max x, e_v = exp(x_v - m),
// Z = sum e_v, p_v = e_v / Z ([P3] SGLang 的实现: softmax(logits / temperature)).
bool softmax_row(const float* row, int32_t V, double T, std::vector<double>& p,
                 double* m_out, double* z_out) {
  p.assign(V, 0.0);
  double m = -std::numeric_limits<double>::infinity();
  for (int32_t v = 0; v < V; ++v) {
    const double x = (double)row[v] / T;
    if (std::isnan(x) || x == std::numeric_limits<double>::infinity()) return false;
    if (x > m) m = x;
  }
  if (m == -std::numeric_limits<double>::infinity()) return false;
  double z = 0.0;
  for (int32_t v = 0; v < V; ++v) {
    p[v] = std::exp((double)row[v] / T - m);
    z += p[v];
  }
  for (int32_t v = 0; v < V; ++v) p[v] /= z;
  *m_out = m;
  *z_out = z;
  return true;
}

// Per-request truncation of one target distribution, in the order of [P3]
// SGLang 的实现 (_sampling_verify): p = softmax(l / T), then top-k
// renormalisation, then top-p renormalisation.
//   top-k (0 < k < V): keep the tokens whose logit is at least the k-th
//     largest logit, counted with multiplicity (every token tied at that value
//     is kept); k <= 0 or k >= V keeps everything;
//   top-p (top_p < 1): of the tokens left, keep those whose renormalised mass
//     strictly above their own probability is below top_p, i.e. the smallest
//     top set whose mass reaches top_p, with ties at its edge kept;
//     top_p >= 1 keeps everything;
// then p' = p restricted to the kept set and renormalised.  Both steps keep a
// set {v : l_v >= tau} (T > 0 keeps the logits' order), and tau, the smallest
// kept logit, is returned.  False for a bad row (as softmax_row).
bool truncate_row(const float* row, int32_t V, double T, int32_t top_k, double top_p,
                  std::vector<double>& p, float* tau_out) {
  double m, z;
  if (!softmax_row(row, V, T, p, &m, &z)) return false;
  std::vector<char> keep(V, 1);
  if (top_k > 0 && top_k < V) {
    std::vector<float> sorted(row, row + V);
    std::sort(sorted.begin(), sorted.end(), [](float a, float b) { return a > b; });
    const float tk = sorted[top_k - 1];
    double s = 0.0;
    for (int32_t v = 0; v < V; ++v) {
      keep[v] = row[v] >= tk;
      if (keep[v]) s += p[v];
    }
    for (int32_t v = 0; v < V; ++v) p[v] = keep[v] ? p[v] / s : 0.0;
  }
  if (top_p < 1.0) {
    // kept tokens by descending logit; a group of equal logits shares the
    // mass strictly above it
    std::vector<int32_t> idx;
    for (int32_t v = 0; v < V; ++v)
      if (keep[v]) idx.push_back(v);
    std::sort(idx.begin(), idx.end(), [&](int32_t a, int32_t b) { return row[a] > row[b]; });
    double above = 0.0;
    size_t i = 0;
    while (i < idx.size()) {
      size_t g = i;
      double gm = 0.0;
      while (g < idx.size() && row[idx[g]] == row[idx[i]]) gm += p[idx[g++]];
      const bool k = above < top_p;
      for (size_t t = i; t < g; ++t) keep[idx[t]] = k;
      above += gm;
      i = g;
    }
    double s = 0.0;
    for (int32_t v = 0; v < V; ++v)
      if (keep[v]) s += p[v];
    for (int32_t v = 0; v < V; ++v) p[v] = keep[v] ? p[v] / s : 0.0;
  }
  float tau = std::numeric_limits<float>::infinity();
  for (int32_t v = 0; v < V; ++v)
    if (keep[v] && row[v] < tau) tau = row[v];
  *tau_out = tau;
  return true;
}

// Smallest v with C_v = r_0 + ... + r_v > t; if rounding leaves C_{V-1} <= t,
// the largest v with r_v > 0.
int32_t sample_cdf(const std::vector<double>& r, double t) {
  double c = 0.0;
  int32_t last_pos = -1;
  for (int32_t v = 0; v < (int32_t)r.size(); ++v) {
    c += r[v];
    if (r[v] > 0.0) last_pos = v;
    if (c > t) return v;
  }
  return last_pos;
}

// Residual of row L ([P2] §2.2): max(0, p - q); one-hot drafts make q the
// indicator of the rejected token ([P3] N-gram 的特殊情况); after all drafts
// are accepted the bonus row has q = 0, so r = p.
void residual(const std::vector<double>& p, const std::vector<double>* q,
              int32_t rejected_token, std::vector<double>& r) {
  const int32_t V = (int32_t)p.size();
  r.assign(V, 0.0);
  for (int32_t v = 0; v < V; ++v) {
    double qv = 0.0;
    if (rejected_token >= 0) qv = q ? (*q)[v] : (v == rejected_token ? 1.0 : 0.0);
    const double d = p[v] - qv;
    r[v] = d > 0.0 ? d : 0.0;
  }
}

}  // namespace

extern "C" {

// ----------------------------- SAM entry points ----------------------------
void* osam_new(int32_t vocab) { return new Sam(vocab); }
void osam_free(void* s) { delete static_cast<Sam*>(s); }

// Extends by n tokens.  Returns 0, or 3 if a token is outside [0, vocab)
// (the automaton is then left as it was before that token).
int32_t osam_extend(void* s, const int32_t* tok, int64_t n) {
  Sam* sam = static_cast<Sam*>(s);
  for (int64_t i = 0; i < n; ++i) {
    if (tok[i] < 0 || tok[i] >= sam->vocab) return 3;
    sam->extend(tok[i]);
  }
  return 0;
}

// info = {draft_len, match_len, min_endpos}
void osam_draft(void* s, int32_t K, int32_t* draft, int32_t* info) {
  static_cast<Sam*>(s)->draft(K, draft, &info[0], &info[1], &info[2]);
}

// sizes = {n_states, n_edges, n_tokens, walk_steps, last}
void osam_sizes(void* s, int64_t* sizes) {
  const Sam* sam = static_cast<Sam*>(s);
  int64_t edges = 0;
  for (const auto& m : sam->next) edges += (int64_t)m.size();
  sizes[0] = (int64_t)sam->len.size();
  sizes[1] = edges;
  sizes[2] = (int64_t)sam->text.size();
  sizes[3] = sam->walk_steps;
  sizes[4] = sam->last;
}

// Copies len/link/min_endpos ([n_states] each) and the edge triples
// (state, token, to) sorted by (state, token) into [n_edges, 3].
void osam_dump(void* s, int32_t* len, int32_t* link, int32_t* min_end, int32_t* edges) {
  const Sam* sam = static_cast<Sam*>(s);
  const size_t ns = sam->len.size();
  for (size_t v = 0; v < ns; ++v) {
    len[v] = sam->len[v];
    link[v] = sam->link[v];
    min_end[v] = sam->min_endpos[v];
  }
  int64_t e = 0;
  for (size_t v = 0; v < ns; ++v)
    for (const auto& kv : sam->next[v]) {
      edges[3 * e + 0] = (int32_t)v;
      edges[3 * e + 1] = kv.first;
      edges[3 * e + 2] = kv.second;
      ++e;
    }
}

// Static matching of one generated text: state[2] = {v, l} is moved by the n
// tokens and the draft of the final state is written (info = {draft_len, l,
// min_endpos of v or -1}).
void osam_match(void* s, int32_t* state, const int32_t* tok, int64_t n, int32_t K, int32_t* draft,
                int32_t* info) {
  const Sam* sam = static_cast<Sam*>(s);
  for (int64_t i = 0; i < n; ++i) sam->match(&state[0], &state[1], tok[i]);
  sam->match_draft(state[0], state[1], K, draft, &info[0]);
  info[1] = state[1];
  info[2] = state[0] != 0 ? sam->min_endpos[state[0]] : -1;
}

// Timing helper: B generated texts matched against one corpus automaton in
// one call (state [B, 2], tokens [B, max_new], n_new [B], draft [B, K],
// info [B, 3]).
void osam_match_batch(void* s, int32_t B, int32_t* state, const int32_t* tokens,
                      const int32_t* n_new, int32_t max_new, int32_t K, int32_t* draft,
                      int32_t* info) {
  for (int32_t b = 0; b < B; ++b)
    osam_match(s, state + 2 * (int64_t)b, tokens + (int64_t)b * max_new, n_new[b], K,
               draft + (int64_t)b * K, info + 3 * (int64_t)b);
}

// Adaptive draft selection between a dynamic and a static automaton ([P4]
// "Drafting with Suffix Automaton"): the dynamic draft is preferred; the
// static one is taken only when its match is longer by more than l_bias.
// Returns 1 if the static draft is chosen.
int32_t oselect_static(int32_t l_static, int32_t l_dynamic, int32_t l_bias) {
  return l_static > l_dynamic + l_bias ? 1 : 0;
}

// Batch helper used for timing: B independent automata, each extended by
// n_new[b] tokens of tokens[b, :] and then drafted.  `handles` holds B
// pointers from osam_new.
void osam_step_batch(void** handles, int32_t B, const int32_t* tokens, const int32_t* n_new,
                     int32_t max_new, int32_t K, int32_t* draft, int32_t* info) {
  for (int32_t b = 0; b < B; ++b) {
    osam_extend(handles[b], tokens + (int64_t)b * max_new, n_new[b]);
    osam_draft(handles[b], K, draft + (int64_t)b * K, info + 3 * (int64_t)b);
  }
}

// ----------------------------- Philox entry points -------------------------
void ophilox4x32_10(const uint32_t* ctr, const uint32_t* key, uint32_t* out) {
  philox4x32_10(ctr, key, out);
}
void ouniforms(uint64_t seed, uint64_t step, int64_t b, int32_t j, double* u) {
  uniforms(seed, step, b, j, &u[0], &u[1]);
}

// ----------------------------- verification --------------------------------
// target:      [B, K+1, V] fp32 logits (bf16 inputs are widened exactly first)
// draftlog:    [B, K, V] fp32 draft logits, or NULL for one-hot drafts
// draft:       [B, K] draft tokens;  draft_len: [B] or NULL (= K for all)
// seq_index:   [B] sequence number fed to the counter, or NULL (= b)
// T == 0 selects greedy verification.
// Outputs [B]: accept_len, out_token, status.  Debug (each may be NULL):
//   row_m, row_z [B, K+1]: m and Z of each evaluated target row (NaN if not
//   evaluated); p_d [B, K+1], q_d [B, K+1]: p_j(d_j), q_j(d_j) of the drafts
//   tested; u_acc [B, K+1]; u_res, res_mass [B]: uniform and sum of the
//   residual used for the final token; row_arg [B, K+1]: greedy argmax.
int32_t over_verify(const float* target, const float* draftlog, const int32_t* draft,
                    const int32_t* draft_len, const int64_t* seq_index, int32_t B, int32_t K,
                    int32_t V, double T, uint64_t seed, uint64_t step, int32_t* accept_len,
                    int32_t* out_token, int32_t* status, double* row_m, double* row_z,
                    double* p_d, double* q_d, double* u_acc, double* u_res, double* res_mass,
                    int32_t* row_arg) {
  const double nan = std::numeric_limits<double>::quiet_NaN();
  std::vector<double> p, q, r;
  for (int32_t b = 0; b < B; ++b) {
    const int64_t sb = seq_index ? seq_index[b] : b;
    const float* trow0 = target + (int64_t)b * (K + 1) * V;
    const float* drow0 = draftlog ? draftlog + (int64_t)b * K * V : nullptr;
    const int32_t* d = draft + (int64_t)b * K;
    for (int32_t j = 0; j <= K; ++j) {
      const int64_t o = (int64_t)b * (K + 1) + j;
      if (row_m) row_m[o] = nan;
      if (row_z) row_z[o] = nan;
      if (p_d) p_d[o] = nan;
      if (q_d) q_d[o] = nan;
      if (u_acc) u_acc[o] = nan;
      if (row_arg) row_arg[o] = -1;
    }
    if (u_res) u_res[b] = nan;
    if (res_mass) res_mass[b] = nan;
    accept_len[b] = -1;
    out_token[b] = -1;
    const int32_t nb = draft_len ? draft_len[b] : K;
    bool bad = nb < 0 || nb > K;
    for (int32_t j = 0; !bad && j < nb; ++j) bad = d[j] < 0 || d[j] >= V;
    if (bad) { status[b] = OV_BADDRAFT; continue; }
    status[b] = OV_OK;

    if (T == 0.0) {
      // greedy: keep the longest prefix of drafts equal to the target argmax,
      // then emit the argmax of the first row that is not accepted.
      int32_t L = nb;
      int32_t a = -1;
      for (int32_t j = 0; j <= nb; ++j) {
        double mv;
        if (!argmax_row(trow0 + (int64_t)j * V, V, &a, &mv)) { status[b] = OV_BADROW; break; }
        const int64_t o = (int64_t)b * (K + 1) + j;
        if (row_m) row_m[o] = mv;
        if (row_arg) row_arg[o] = a;
        if (j == nb || d[j] != a) { L = j; break; }
      }
      if (status[b] != OV_OK) continue;
      accept_len[b] = L;
      out_token[b] = a;
      continue;
    }

    // rejection sampling: accept d_j iff u_j * q_j(d_j) <= p_j(d_j), i.e.
    // u_j <= min(1, p/q) ([P1] §1.1 eps <= alpha(x); [P2] §2.2)
    int32_t L = nb;
    bool ok = true;
    for (int32_t j = 0; j <= nb; ++j) {
      double m, z;
      const int64_t o = (int64_t)b * (K + 1) + j;
      if (!softmax_row(trow0 + (int64_t)j * V, V, T, p, &m, &z)) { ok = false; break; }
      if (row_m) row_m[o] = m;
      if (row_z) row_z[o] = z;
      if (j == nb) { L = nb; break; }  // every draft accepted: bonus row
      double qd = 1.0;
      if (drow0) {
        double mq, zq;
        if (!softmax_row(drow0 + (int64_t)j * V, V, T, q, &mq, &zq)) { ok = false; break; }
        qd = q[d[j]];
      }
      double ua, ur;
      uniforms(seed, step, sb, j, &ua, &ur);
      if (p_d) p_d[o] = p[d[j]];
      if (q_d) q_d[o] = qd;
      if (u_acc) u_acc[o] = ua;
      if (!(ua * qd <= p[d[j]])) { L = j; break; }
    }
    if (!ok) { status[b] = OV_BADROW; continue; }
    // p holds row L's target distribution; q holds row L's draft distribution
    // when draft logits are given and L < nb.
    const bool rejected = L < nb;
    residual(p, (drow0 && rejected) ? &q : nullptr, rejected ? d[L] : -1, r);
    double mass = 0.0;
    for (int32_t v = 0; v < V; ++v) mass += r[v];
    if (!(mass > 0.0)) {  // cannot happen in exact arithmetic: fall back to p
      r = p;
      mass = 0.0;
      for (int32_t v = 0; v < V; ++v) mass += r[v];
    }
    double ua, ur;
    uniforms(seed, step, sb, L, &ua, &ur);
    accept_len[b] = L;
    out_token[b] = sample_cdf(r, ur * mass);
    if (u_res) u_res[b] = ur;
    if (res_mass) res_mass[b] = mass;
  }
  return 0;
}

// Tree verification ([P3] SGLang 的实现: the candidates of a draft tree are
// tried sibling by sibling, one coin per depth against the running sum of
// their target probabilities; a rejected candidate's probability is removed
// before the final sample; [P3] N-gram 的特殊情况: model-free candidates have
// q = 0).  Sequence b's tree has N nodes: node 0 is the verified context,
// node n >= 1 carries token tok[n]; first_child / next_sibling link them
// (-1: none), each link pointing to a larger node index, each node n >= 1
// linked exactly once, siblings carrying distinct tokens.  Row n of target
// ([B, N, V]) scores the token after node n's path.
//   greedy (T = 0): at node c follow the child whose token is the row's
//     argmax; stop at the first node without such a child and emit that
//     argmax;
//   sampling: at node c with children k_1 .. k_m (in sibling order) draw
//     u = U_acc(depth); take k_i for the first i with u <= p(k_1) + ... +
//     p(k_i); if there is none, or c has no children, stop and emit a token
//     drawn from p_c with the tried children's probabilities set to 0, by
//     t = U_res(depth) * (remaining mass).  Whatever the tree, the emitted
//     tokens follow the target distribution.
// Outputs: accept_len (depth reached), out_token, path [B, N] (accepted node
// indices, -1 after), status (BADDRAFT for a malformed tree, BADROW).
int32_t over_tree_verify(const float* target, const int32_t* tok, const int32_t* first_child,
                         const int32_t* next_sibling, int32_t B, int32_t N, int32_t V, double T,
                         uint64_t seed, uint64_t step, int32_t* accept_len, int32_t* out_token,
                         int32_t* path, int32_t* status, double* u_res, double* res_mass) {
  std::vector<double> p, r;
  std::vector<int32_t> refs;
  for (int32_t b = 0; b < B; ++b) {
    const float* rows = target + (int64_t)b * N * V;
    const int32_t* tk = tok + (int64_t)b * N;
    const int32_t* fc = first_child + (int64_t)b * N;
    const int32_t* ns = next_sibling + (int64_t)b * N;
    int32_t* pb = path + (int64_t)b * N;
    for (int32_t n = 0; n < N; ++n) pb[n] = -1;
    accept_len[b] = -1;
    out_token[b] = -1;
    if (u_res) u_res[b] = std::numeric_limits<double>::quiet_NaN();
    if (res_mass) res_mass[b] = std::numeric_limits<double>::quiet_NaN();
    // the tree's shape
    bool bad = N < 1 || ns[0] != -1;
    refs.assign(N, 0);
    for (int32_t n = 0; !bad && n < N; ++n) {
      if (n > 0 && (tk[n] < 0 || tk[n] >= V)) bad = true;
      for (int32_t l : {fc[n], ns[n]}) {
        if (l == -1) continue;
        if (l <= n || l >= N) bad = true;
        else ++refs[l];
      }
    }
    for (int32_t n = 1; !bad && n < N; ++n) bad = refs[n] != 1;
    for (int32_t n = 0; !bad && n < N; ++n)
      for (int32_t a = fc[n]; !bad && a != -1; a = ns[a])
        for (int32_t c = ns[a]; !bad && c != -1; c = ns[c]) bad = tk[a] == tk[c];
    if (bad) {
      status[b] = OV_BADDRAFT;
      continue;
    }
    status[b] = OV_OK;
    int32_t cur = 0, depth = 0;
    if (T == 0.0) {
      for (;;) {
        int32_t a;
        double mv;
        if (!argmax_row(rows + (int64_t)cur * V, V, &a, &mv)) {
          status[b] = OV_BADROW;
          break;
        }
        int32_t next = -1;
        for (int32_t c = fc[cur]; c != -1; c = ns[c])
          if (tk[c] == a) next = c;
        if (next == -1) {
          accept_len[b] = depth;
          out_token[b] = a;
          break;
        }
        pb[depth++] = next;
        cur = next;
      }
      continue;
    }
    for (;;) {
      double m, z;
      if (!softmax_row(rows + (int64_t)cur * V, V, T, p, &m, &z)) {
        status[b] = OV_BADROW;
        break;
      }
      double ua, ur;
      uniforms(seed, step, b, depth, &ua, &ur);
      int32_t next = -1;
      double acc = 0.0;
      r = p;
      for (int32_t c = fc[cur]; c != -1; c = ns[c]) {
        acc += p[tk[c]];
        if (ua <= acc) {
          next = c;
          break;
        }
        r[tk[c]] = 0.0;  // tried and rejected: out of the final distribution
      }
      if (next != -1) {
        pb[depth++] = next;
        cur = next;
        continue;
      }
      double mass = 0.0;
      for (int32_t v = 0; v < V; ++v) mass += r[v];
      if (!(mass > 0.0)) {  // cannot happen in exact arithmetic: fall back to p
        r = p;
        mass = 1.0;
      }
      accept_len[b] = depth;
      out_token[b] = sample_cdf(r, ur * mass);
      if (u_res) u_res[b] = ur;
      if (res_mass) res_mass[b] = mass;
      break;
    }
  }
  return 0;
}

// For parity checks of tree verification at one node: acc[i] = p(k_1) + ...
// + p(k_{i+1}) for the n children tokens (sibling order), and the interval
// [lo, hi) of `token` in the node's final-sample distribution (the row
// without the children, normalised) -- lo_hi_mass = {lo, hi, mass}.
void over_tree_node_info(const float* trow, int32_t V, double T, const int32_t* children,
                         int32_t n, int32_t token, double* acc, double* lo_hi_mass) {
  std::vector<double> p;
  double m, z;
  softmax_row(trow, V, T, p, &m, &z);
  double a = 0.0;
  std::vector<double> r = p;
  for (int32_t i = 0; i < n; ++i) {
    a += p[children[i]];
    acc[i] = a;
    r[children[i]] = 0.0;
  }
  double mass = 0.0;
  for (int32_t v = 0; v < V; ++v) mass += r[v];
  double before = 0.0;
  for (int32_t v = 0; v < token; ++v) before += r[v];
  lo_hi_mass[0] = before / mass;
  lo_hi_mass[1] = (before + r[token]) / mass;
  lo_hi_mass[2] = mass;
}

// Normalised CDF interval [lo, hi) of `token` under the residual of one row:
// lo = C_{token-1} / sum r, hi = C_token / sum r.  Used by the parity tests to
// decide whether a differing resample lies within a rounding band of a CDF
// boundary.  rejected_token < 0 selects the bonus residual (r = p).
void over_cdf_interval(const float* trow, const float* drow, int32_t V, double T,
                       int32_t rejected_token, int32_t token, double* lo_hi_mass) {
  std::vector<double> p, q, r;
  double m, z;
  softmax_row(trow, V, T, p, &m, &z);
  if (drow && rejected_token >= 0) softmax_row(drow, V, T, q, &m, &z);
  residual(p, (drow && rejected_token >= 0) ? &q : nullptr, rejected_token, r);
  double mass = 0.0;
  for (int32_t v = 0; v < V; ++v) mass += r[v];
  double c = 0.0, lo = 0.0;
  for (int32_t v = 0; v <= token && v < V; ++v) {
    lo = c;
    c += r[v];
  }
  lo_hi_mass[0] = lo / mass;
  lo_hi_mass[1] = c / mass;
  lo_hi_mass[2] = mass;
}

// Verification with per-request sampling parameters ([P3] SGLang 的实现,
// _sampling_verify: per-request temperature, top_k and top_p applied to the
// target probabilities before the drafts are tested; [P3] N-gram 的特殊情况:
// one-hot drafts).  Row j's distribution is p'_j = truncate_row(row j, T_b,
// k_b, top_p_b); d_j is accepted iff u_j <= p'_j(d_j); the final token is
// drawn by u' from max(0, p'_L - 1[d_L]) after a rejection, or from p'_L for
// the bonus row (the same residual rule as over_verify).
// temp, top_k, top_p: [B].  Outputs as over_verify, plus tau [B, K+1] (the
// smallest kept logit of each evaluated row, NaN otherwise; may be NULL).
int32_t over_verify_sampling(const float* target, const int32_t* draft, const int32_t* draft_len,
                             int32_t B, int32_t K, int32_t V, const double* temp,
                             const int32_t* top_k, const double* top_p, uint64_t seed,
                             uint64_t step, int32_t* accept_len, int32_t* out_token,
                             int32_t* status, double* p_d, double* u_acc, double* u_res,
                             double* res_mass, float* tau) {
  const double nan = std::numeric_limits<double>::quiet_NaN();
  std::vector<double> p, r;
  for (int32_t b = 0; b < B; ++b) {
    const float* trow0 = target + (int64_t)b * (K + 1) * V;
    const int32_t* d = draft + (int64_t)b * K;
    for (int32_t j = 0; j <= K; ++j) {
      const int64_t o = (int64_t)b * (K + 1) + j;
      if (p_d) p_d[o] = nan;
      if (u_acc) u_acc[o] = nan;
      if (tau) tau[o] = std::numeric_limits<float>::quiet_NaN();
    }
    if (u_res) u_res[b] = nan;
    if (res_mass) res_mass[b] = nan;
    accept_len[b] = -1;
    out_token[b] = -1;
    const int32_t nb = draft_len ? draft_len[b] : K;
    bool bad = nb < 0 || nb > K;
    for (int32_t j = 0; !bad && j < nb; ++j) bad = d[j] < 0 || d[j] >= V;
    if (bad) { status[b] = OV_BADDRAFT; continue; }
    const double T = temp[b], tp = top_p[b];
    if (!(T > 0.0) || T == std::numeric_limits<double>::infinity() || !(tp > 0.0)) {
      status[b] = OV_BADPARAM;
      continue;
    }
    status[b] = OV_OK;
    int32_t L = nb;
    bool ok = true;
    for (int32_t j = 0; j <= nb; ++j) {
      const int64_t o = (int64_t)b * (K + 1) + j;
      float tj;
      if (!truncate_row(trow0 + (int64_t)j * V, V, T, top_k[b], tp, p, &tj)) { ok = false; break; }
      if (tau) tau[o] = tj;
      if (j == nb) { L = nb; break; }
      double ua, ur;
      uniforms(seed, step, b, j, &ua, &ur);
      if (p_d) p_d[o] = p[d[j]];
      if (u_acc) u_acc[o] = ua;
      if (!(ua <= p[d[j]])) { L = j; break; }
    }
    if (!ok) { status[b] = OV_BADROW; continue; }
    const bool rejected = L < nb;
    residual(p, nullptr, rejected ? d[L] : -1, r);
    double mass = 0.0;
    for (int32_t v = 0; v < V; ++v) mass += r[v];
    if (!(mass > 0.0)) {  // only the rejected token was kept: sample p' itself
      r = p;
      mass = 0.0;
      for (int32_t v = 0; v < V; ++v) mass += r[v];
    }
    double ua, ur;
    uniforms(seed, step, b, L, &ua, &ur);
    accept_len[b] = L;
    out_token[b] = sample_cdf(r, ur * mass);
    if (u_res) u_res[b] = ur;
    if (res_mass) res_mass[b] = mass;
  }
  return 0;
}

// One row through truncate_row: p' into p_out [V], the smallest kept logit
// into tau_out[0]; returns 0, or OV_BADROW.
int32_t over_truncate_row(const float* row, int32_t V, double T, int32_t top_k, double top_p,
                          double* p_out, float* tau_out) {
  std::vector<double> p;
  if (!truncate_row(row, V, T, top_k, top_p, p, tau_out)) return OV_BADROW;
  for (int32_t v = 0; v < V; ++v) p_out[v] = p[v];
  return 0;
}

}  // extern "C"

