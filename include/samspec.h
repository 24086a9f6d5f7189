/*
 * samspec.h -- C ABI of libsamspec.so: device-resident dynamic suffix automata
 * (D-SAM) for model-free drafting, and lossless speculative verification.
 *
 * Pages the operations come from (titles as printed, with the section):
 *   [P1] "SAM投机推理：长序列强化学习训练加速利器" (CANN cann-recipes-train)
 *        §1.1 SAM 原理 -- endpos, link, next, dynamic SAM updated after each
 *        verified token, min_endpos, draft by walking link edges (ABCBC
 *        example), rejection test eps <= alpha(x); §3.1.2 拒绝采样加速 --
 *        recovered-token sampling and the accept/reject chain.
 *   [P2] nxbn.cn speculative-sampling article, §2.2 验证阶段的并行打分机制 --
 *        accept with probability min(1, p_target/p_draft), resample from the
 *        positive part of (p_target - p_draft), K+1 distributions per pass.
 *   [P3] gogongxt.com notes "投机采样": 贪婪采样 (greedy), 拒绝采样, SGLang 的实现
 *        (softmax(logits / temperature)), N-gram 的特殊情况 (draft_probs = 0).
 *   [P4] volcengine.com SAM-Decoding article, §3 Suffix Automaton Construction,
 *        Drafting with Suffix Automaton, Update of Suffix Automaton.
 *
 * Conventions for every entry point:
 *   - d_ pointers are DEVICE pointers, h_ pointers HOST pointers.
 *   - The caller owns all memory.  The library never allocates device memory;
 *     it lays its state out inside a caller-provided workspace.  Host-side
 *     descriptors (sam_batch) are malloc'd by sam_batch_create and freed by
 *     sam_batch_destroy.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) unless it says it synchronises.  Inputs are read only;
 *     only the named outputs and the batch's own workspace are written.
 *   - Return value: SAMSPEC_OK (0) or a negative host-side error, detected
 *     synchronously before any launch (arguments, sizes, alignment) or from
 *     the launch itself (SAMSPEC_ECUDA).  Conditions found on the device are
 *     reported per sequence through status words (positive codes below); a
 *     sequence with a non-zero SAM status is frozen (no further extension,
 *     draft_len 0) while the other sequences proceed.  Nothing traps.
 *   - All lengths and positions are 0-based token counts.
 */
#ifndef SAMSPEC_H_
#define SAMSPEC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Type-compatible with cudaStream_t; avoids requiring the CUDA headers. */
typedef struct CUstream_st* samspec_stream_t;

/* ---- host-side return codes ---- */
#define SAMSPEC_OK 0
#define SAMSPEC_EINVAL (-1)  /* null pointer, negative size, bad argument     */
#define SAMSPEC_ESIZE (-2)   /* a size above a documented limit / workspace   */
#define SAMSPEC_EDTYPE (-3)  /* unknown logits dtype                          */
#define SAMSPEC_ECUDA (-4)   /* a CUDA runtime call or launch failed          */
#define SAMSPEC_EALIGN (-5)  /* a pointer below its documented alignment      */

/* ---- per-sequence device status words ---- */
#define SAMSPEC_ST_OK 0
#define SAMSPEC_ST_CAPACITY 1  /* token, state or edge capacity exhausted      */
#define SAMSPEC_ST_HASHFULL 2  /* transition hash found no free slot           */
#define SAMSPEC_ST_TOKEN 3     /* a token outside [0, vocab)                   */
#define SAMSPEC_ST_LOOPCAP 4   /* a link walk exceeded its bound (corruption)  */
#define SAMSPEC_ST_BADROW 5    /* verify: a needed row has NaN, or (T > 0) a   */
                               /* +inf, or is entirely -inf                    */
#define SAMSPEC_ST_BADDRAFT 6  /* verify: draft_len outside [0, K] or a draft  */
                               /* token outside [0, V); extend: n_new outside  */
                               /* [0, max_new]                                 */
#define SAMSPEC_ST_TIMEOUT 7   /* verify: a bounded on-chip wait ran out       */
#define SAMSPEC_ST_BADPARAM 8  /* verify with sampling parameters: temperature  */
                               /* not > 0 and finite, or top_p not > 0         */
#define SAMSPEC_ST_BOUNDS 9    /* automata, debug library only (built with     */
                               /* SAMSPEC_CHECKS=1): an index into one of the  */
                               /* sequence's arrays fell outside the array; the */
                               /* access was skipped and the sequence frozen   */

/* logits element types */
#define SAMSPEC_F32 0
#define SAMSPEC_BF16 1

/* Library version (major * 10000 + minor * 100 + patch). */
int samspec_version(void);
/* Static string for any return code or status word. */
const char* samspec_strerror(int code);

/* =========================================================================
 * Dynamic suffix automata, one per sequence ([P1] §1.1 动态 SAM; [P4] §3).
 *
 * Each sequence b owns the automaton of its text S_b = s_0 ... s_{n-1}
 * (prompt followed by every appended token).  States carry len (longest
 * string), link (suffix link, -1 at the root = state 0) and min_endpos (the
 * smallest end position of the state's strings, [P4] §3); transitions live in
 * an open-addressed (state, token) -> state hash.  States are numbered in
 * creation order, a split's new state before its clone, so the arrays are
 * identical to those of a plain sequential construction.
 *
 * Capacities per sequence for capacity_tokens = C: C tokens, 2C + 1 states,
 * 3C + 4 transitions (each state's out-tokens kept in a contiguous array of
 * a pool of 4 x (3C + 4) ints), and a power-of-two hash of at least
 * 1.5 x (3C + 4) slots.  Limits: 1 <= B <= 2^20, 1 <= C <= 2^22 - 1, 1 <= vocab <= 2^18.
 * ========================================================================= */
typedef struct sam_batch sam_batch;

/* Bytes of device workspace sam_batch_create needs for (B, C).  Returns 0 for
 * arguments outside the limits above. */
size_t sam_batch_workspace_bytes(int32_t B, int32_t capacity_tokens);

/* Lays out B empty automata in d_workspace (256-byte aligned, at least
 * sam_batch_workspace_bytes(B, C) bytes, owned by the caller and kept alive
 * until sam_batch_destroy) and enqueues their initialisation on `stream`.
 * *out receives a host descriptor.  Errors: EINVAL, ESIZE, EALIGN, ECUDA. */
int sam_batch_create(int32_t B, int32_t capacity_tokens, int32_t vocab, void* d_workspace,
                     size_t ws_bytes, samspec_stream_t stream, sam_batch** out);

/* Frees the host descriptor only (never the caller's workspace). */
int sam_batch_destroy(sam_batch* batch);

/* Empties the automata of the sequences with d_seq_mask[b] != 0 (all of them
 * when d_seq_mask is NULL) and clears their status.  Asynchronous. */
int sam_reset(sam_batch* batch, const int32_t* d_seq_mask, samspec_stream_t stream);

/* Appends tokens to every sequence ([P1] §1.1: the D-SAM is extended by each
 * token the target model has verified; [P4] Update of Suffix Automaton).
 *   d_tokens: [B, max_new] int32 row-major; row b holds sequence b's tokens.
 *   d_n_new:  [B] int32, 0 <= n_new[b] <= max_new tokens taken from row b.
 * A bulk prompt build (prefill) is the same call with a long max_new.
 * Device errors per sequence: ST_TOKEN, ST_CAPACITY, ST_HASHFULL,
 * ST_LOOPCAP, ST_BADDRAFT (n_new out of range).  Asynchronous. */
int sam_extend(sam_batch* batch, const int32_t* d_tokens, const int32_t* d_n_new,
               int32_t max_new, samspec_stream_t stream);

/* Draft query ([P1] §1.1 草稿生成; [P4] Drafting with Suffix Automaton).
 * From the state of S_b follow link edges to the first state v that has an
 * outgoing transition; v's longest string is the longest suffix of S_b that
 * also ends earlier in S_b.  With e = min_endpos(v):
 *   d_draft[b, t]   = s_{e+1+t} for t < draft_len, -1 after   ([B, K] int32)
 *   d_draft_len[b]  = min(K, n - 1 - e), 0 when v is the root  ([B] int32)
 *   d_match_len[b]  = len(v) (0 at the root)                   ([B] int32)
 *   d_min_endpos[b] = e (-1 at the root)                        ([B] int32)
 * d_draft_len, d_match_len and d_min_endpos may be NULL.  A frozen sequence
 * reports draft_len 0.  1 <= K <= 64.  Asynchronous. */
int sam_draft(sam_batch* batch, int32_t K, int32_t* d_draft, int32_t* d_draft_len,
              int32_t* d_match_len, int32_t* d_min_endpos, samspec_stream_t stream);

/* sam_extend followed by sam_draft in one launch (the per-step update of
 * [P4]: extend with the accepted tokens, then move to the new matching state
 * and draft).  Same arguments and semantics as the two calls. */
int sam_step(sam_batch* batch, const int32_t* d_tokens, const int32_t* d_n_new,
             int32_t max_new, int32_t K, int32_t* d_draft, int32_t* d_draft_len,
             int32_t* d_match_len, int32_t* d_min_endpos, samspec_stream_t stream);

/* sam_step on n sequences of the batch: call index i (0 <= i < n) works on
 * automaton d_rows[i] (d_rows NULL: automaton i, n <= B); d_tokens [n, max_new],
 * d_n_new [n] and the draft outputs [n, K] / [n] follow the call index, so a
 * caller can pass only its active sequences.  K = 0 extends without drafting
 * (d_draft may be NULL; d_draft_len, if given, is set to 0; match_len and
 * min_endpos are not written).
 * Rows must be distinct within a call; a row outside [0, B) leaves no
 * automaton changed and gets an empty draft. */
int sam_step_rows(sam_batch* batch, const int32_t* d_rows, int32_t n, const int32_t* d_tokens,
                  const int32_t* d_n_new, int32_t max_new, int32_t K, int32_t* d_draft,
                  int32_t* d_draft_len, int32_t* d_match_len, int32_t* d_min_endpos,
                  samspec_stream_t stream);

/* Static use of an automaton ([P4] "Drafting with Suffix Automaton",
 * "Update of Suffix Automaton"; [P1] §1.1 静态 SAM): automaton `corpus_row` of
 * `corpus` holds a corpus (documents joined by an end-of-sequence token,
 * built with sam_extend) and is only read.  Call index i follows a generated
 * text with the matching state d_state[2i], d_state[2i+1] = {state, length}
 * of its longest suffix that occurs in the corpus ({0, 0} to start); the
 * n_new[i] tokens d_tokens[i, :] move it along (a transition from the state,
 * else from the first state on its suffix chain that has one, else to
 * {0, 0}).  Then K corpus tokens after the state's min_endpos are drafted
 * into d_draft [n, K] (-1 padded; d_draft_len [n]); d_match_len [n] and
 * d_min_endpos [n] receive the length and that position (-1 at the root).
 * A token outside [0, vocab) resets the state to {0, 0}.  The corpus is not
 * modified, so any number of calls may read it at once.  One launch. */
int ssam_match(const sam_batch* corpus, int32_t corpus_row, int32_t n, int32_t* d_state,
               const int32_t* d_tokens, const int32_t* d_n_new, int32_t max_new, int32_t K,
               int32_t* d_draft, int32_t* d_draft_len, int32_t* d_match_len,
               int32_t* d_min_endpos, samspec_stream_t stream);

/* Adaptive choice between a dynamic and a static automaton's drafts ([P4]
 * "Drafting with Suffix Automaton": the dynamic draft is preferred): per
 * sequence, the static draft (d_st_*) is taken when its match length exceeds
 * the dynamic one (d_dyn_*) by more than l_bias, else the dynamic draft.
 * Writes d_draft [n, K], d_draft_len [n] and, optionally, d_source [n]
 * (1 = static).  One launch. */
int sam_select_drafts(int32_t n, int32_t K, const int32_t* d_dyn_draft, const int32_t* d_dyn_len,
                      const int32_t* d_dyn_match, const int32_t* d_st_draft,
                      const int32_t* d_st_len, const int32_t* d_st_match, int32_t l_bias,
                      int32_t* d_draft, int32_t* d_draft_len, int32_t* d_source,
                      samspec_stream_t stream);

/* Copies the B status words to h_status[B] (host memory) and synchronises
 * `stream`. */
int sam_get_status(sam_batch* batch, int32_t* h_status, samspec_stream_t stream);

/* Snapshot / restore of the whole batch: d_dst / d_src must hold
 * sam_batch_workspace_bytes(B, C) bytes.  Asynchronous device-to-device copy. */
int sam_export(sam_batch* batch, void* d_dst, size_t bytes, samspec_stream_t stream);
int sam_import(sam_batch* batch, const void* d_src, size_t bytes, samspec_stream_t stream);

/* Inspection hook (synchronises `stream`): copies sequence b's automaton to
 * host memory.  h_scalars[8] = {n_tokens, last, n_states, n_edges, status,
 * link(last), 0, 0}; h_len/h_link/h_min_endpos receive up to max_states
 * entries; h_edges receives up to max_edges (state, token, to) triples,
 * sorted by (state, token).  Any h_ array may be NULL. */
int sam_dump_sequence(sam_batch* batch, int32_t b, int32_t* h_scalars, int32_t* h_len,
                      int32_t* h_link, int32_t* h_min_endpos, int32_t max_states,
                      int32_t* h_edges, int32_t max_edges, samspec_stream_t stream);

/* =========================================================================
 * Lossless verification of K drafts per sequence ([P2] §2.2; [P3] 贪婪采样,
 * 拒绝采样, SGLang 的实现, N-gram 的特殊情况; [P1] §1.1, §3.1.2).
 *
 *   d_target       [B, K+1, V] logits (SAMSPEC_F32 or SAMSPEC_BF16), row-major,
 *                  V contiguous; row j scores the token after draft j-1.
 *   d_draft_logits [B, K, V] logits of a draft model, or NULL for one-hot
 *                  drafts (a suffix automaton's draft has q = indicator).
 *   d_draft        [B, K] int32 draft tokens d_0 .. d_{K-1} (may be NULL when
 *                  K = 0: no drafts, the bonus row alone is sampled).
 *   d_draft_len    [B] int32 n_b in [0, K], or NULL (n_b = K).
 *   temperature    0 selects greedy verification: accept while d_j equals
 *                  the row's argmax (lowest id on ties); the emitted token is
 *                  the argmax of the first non-accepted row.
 *                  T > 0: p_j = softmax(target_j / T), q_j = softmax(draft_j / T)
 *                  or one-hot at d_j; accept d_j iff u_j * q_j(d_j) <= p_j(d_j);
 *                  L = first rejected j (or n_b); the emitted token is drawn
 *                  from r = max(0, p_L - q_L) (bonus row L = n_b: r = p_L) as
 *                  the smallest id whose running sum of r exceeds u'_L * sum(r).
 *   seed, step     key and counter of Philox4x32-10: u_j / u'_j are words 0 / 1
 *                  of Philox(key = (seed lo, seed hi), counter = (j, b, step lo,
 *                  step hi)) mapped by U(x) = ((x >> 9) + 0.5) * 2^-23.
 * Outputs (device, [B] int32):
 *   d_accept_len   L (-1 for a sequence with a non-zero status)
 *   d_out_token    the bonus or resampled token (-1 on error)
 *   d_emit         optional [B, K+1]: d_0 .. d_{L-1}, out_token, then -1
 *   d_emit_len     optional [B]: L + 1 (0 on error)
 *   d_status       optional [B]: ST_OK, ST_BADROW, ST_BADDRAFT or ST_TIMEOUT
 *   dbg            optional device pointers (any may be NULL), [B, K+1] fp32
 *                  unless noted, written only for rows the chain evaluated:
 *                  row_m (T > 0: max_v l_v / T; T = 0: max_v l_v), row_z
 *                  (sum_v exp(l_v / T - row_m)), p_d (p_j(d_j)), q_d (q_j(d_j)),
 *                  row_arg (int32 argmax, greedy); res_mass [B] (sum r over the
 *                  final row, in units of p).
 * Workspace: d_workspace of spec_verify_workspace_bytes(B, K, V) bytes,
 * 256-byte aligned, zeroed once with spec_verify_workspace_init before first
 * use and not shared by two calls in flight.  Logits pointers must be 16-byte
 * aligned.  Limits: 1 <= B <= 2^24, 0 <= K <= 32, and V at most 48 tiles of
 * the kernel's 48 KB staging buffer with one-hot drafts (or greedy), 32 tiles
 * with draft logits (T > 0): 589824 (fp32 target, greedy or one-hot drafts),
 * 1179648 (bf16 target, greedy or one-hot), 393216 (bf16 target and bf16 draft
 * logits), 196608 (any other pair with draft logits); larger V returns
 * SAMSPEC_ESIZE.  Asynchronous; one kernel launch. */
typedef struct spec_verify_debug {
  float* row_m;
  float* row_z;
  float* p_d;
  float* q_d;
  int32_t* row_arg;
  float* res_mass;
} spec_verify_debug;

size_t spec_verify_workspace_bytes(int32_t B, int32_t K, int32_t V);
int spec_verify_workspace_init(void* d_workspace, size_t ws_bytes, samspec_stream_t stream);

int spec_verify(const void* d_target, int32_t target_dtype, const void* d_draft_logits,
                int32_t draft_dtype, const int32_t* d_draft, const int32_t* d_draft_len,
                int32_t B, int32_t K, int32_t V, float temperature, uint64_t seed, uint64_t step,
                int32_t* d_accept_len, int32_t* d_out_token, int32_t* d_emit,
                int32_t* d_emit_len, int32_t* d_status, const spec_verify_debug* dbg,
                void* d_workspace, size_t ws_bytes, samspec_stream_t stream);

/* spec_verify for callers that cannot allocate device memory: code running
 * where cudaMalloc is off limits (a host framework that owns every device
 * allocation through its own pool, a plugin loaded into such a runtime, or a
 * caller in a context where allocating would synchronise the device).  The
 * method's pages have no counterpart; it is a convenience of this library.
 *
 * Same arguments, outputs and limits as spec_verify, without the workspace:
 * its scratch (the kernel's work counters) is a fixed 256-byte array inside
 * the library, present on every device that loads it until the process
 * exits.  Every size spec_verify takes fits that array, so the limits are
 * spec_verify's (1 <= B <= 2^24, 0 <= K <= 32, V within the tile limits
 * above); anything beyond them returns SAMSPEC_ESIZE, and every argument
 * error is returned before anything is enqueued.  The call allocates
 * nothing: it clears the array with cudaMemsetAsync on `stream` and launches
 * the same kernel as spec_verify.
 *   - The first call on a device looks the array's device address up (with
 *     that device current) and caches it; make that first call before any
 *     stream capture.  After cudaDeviceReset of a device the cached address
 *     is stale: do not call this entry point on that device again in the
 *     same process.
 *   - All calls on a device share the one array: two calls whose kernels
 *     overlap on the GPU (different streams, no ordering between them) race
 *     on it and give wrong results.  Serialise them, or use spec_verify with
 *     a workspace each. */
int spec_verify_noalloc(const void* d_target, int32_t target_dtype, const void* d_draft_logits,
                        int32_t draft_dtype, const int32_t* d_draft, const int32_t* d_draft_len,
                        int32_t B, int32_t K, int32_t V, float temperature, uint64_t seed,
                        uint64_t step, int32_t* d_accept_len, int32_t* d_out_token,
                        int32_t* d_emit, int32_t* d_emit_len, int32_t* d_status,
                        const spec_verify_debug* dbg, samspec_stream_t stream);

/* Verification of a draft tree per sequence ([P3] SGLang 的实现: candidates
 * are tried sibling by sibling; [P3] N-gram 的特殊情况: model-free drafts have
 * q = 0).  Sequence b's tree has N nodes (1 <= N <= 32): node 0 is the
 * verified context, node n >= 1 carries token d_tok[b, n]; d_first_child and
 * d_next_sibling [B, N] link them (-1: none).  Every link must point to a
 * larger index below N, every node n >= 1 must be linked exactly once, node 0
 * has no sibling, tokens lie in [0, V) and siblings carry distinct tokens;
 * otherwise the sequence gets ST_BADDRAFT.  d_target [B, N, V]: row n scores
 * the token after node n's path.
 *   T = 0: at each node the child whose token is the row's argmax is taken;
 *          the first node without one emits its argmax.
 *   T > 0: at depth t a coin u_t (Philox word 0 of counter (t, b, step))
 *          takes the first child k_i (sibling order) with
 *          u_t <= p(k_1) + ... + p(k_i); with none, or at a leaf, the emitted
 *          token is drawn from p of the node with the tried children removed,
 *          by u'_t (word 1) as in spec_verify.  A tree of one child per node
 *          is the linear case of spec_verify.
 * Outputs: d_accept_len [B] (depth reached), d_out_token [B], optional
 * d_path [B, N] (accepted node indices, -1 after), d_emit [B, N] (their tokens,
 * then the emitted token, -1 after), d_emit_len, d_status; dbg row_m / row_z /
 * row_arg / res_mass as for spec_verify (rows indexed by node; p_d and q_d
 * are not written).  Workspace as spec_verify_workspace_bytes(B, N - 1, V).
 * V limits as spec_verify's one-hot case.  One kernel launch. */
int spec_verify_tree(const void* d_target, int32_t target_dtype, const int32_t* d_tok,
                     const int32_t* d_first_child, const int32_t* d_next_sibling, int32_t B,
                     int32_t N, int32_t V, float temperature, uint64_t seed, uint64_t step,
                     int32_t* d_accept_len, int32_t* d_out_token, int32_t* d_path,
                     int32_t* d_emit, int32_t* d_emit_len, int32_t* d_status,
                     const spec_verify_debug* dbg, void* d_workspace, size_t ws_bytes,
                     samspec_stream_t stream);

/* The cut of each target row under per-request sampling parameters ([P3]
 * SGLang 的实现, _sampling_verify: p = softmax(l / T), then top-k
 * renormalisation, then top-p renormalisation).  For row (b, r) of d_target
 * [B, R, V] (1 <= R <= 33, V <= 2^21, 16-byte aligned) with d_temperature[b],
 * d_top_k[b], d_top_p[b] ([B] each, device):
 *   top-k (0 < k < V) keeps the tokens whose logit is at least the k-th
 *   largest (ties kept); top-p (top_p < 1) keeps, of those, the ones whose
 *   mass strictly above them is below top_p of their total (the smallest top
 *   set reaching top_p, ties kept).  Both keep {v : l_v >= tau};
 * d_tau [B, R] receives tau (fp32): -inf when nothing is cut (k <= 0 or
 * k >= V, and top_p >= 1) or the row has NaN, +inf or only -inf logits; NaN
 * when T is not > 0 and finite or top_p is not > 0.  Masses are summed
 * exactly in fixed point, each term floored to units of 2^-42 of the row
 * maximum's term, so a top-p cut whose mass lies within V * 2^-42 of top_p
 * (under 5e-7 at V = 2^21) may fall on either side.  fp32 rows: one launch;
 * bf16 rows: two (the second cuts only rows holding more than 65,535 equal
 * logits).  Asynchronous. */
int spec_sampling_cut(const void* d_target, int32_t target_dtype, int32_t B, int32_t R, int32_t V,
                      const float* d_temperature, const int32_t* d_top_k, const float* d_top_p,
                      float* d_tau, samspec_stream_t stream);

/* Verification with per-request sampling parameters ([P3] SGLang 的实现: the
 * target probabilities are softmax(l / T_b), top-k renormalised, then top-p
 * renormalised before the drafts are tested; [P3] N-gram 的特殊情况: one-hot
 * drafts).  As spec_verify at T > 0 with one-hot drafts, except that
 * sequence b uses d_temperature[b] and row j of it the truncated
 * distribution p'_j (spec_sampling_cut's tau; logits below it have
 * probability 0): d_j is accepted iff u_j <= p'_j(d_j); the final token is
 * drawn from p'_L without d_L after a rejection, or from p'_L for the bonus
 * row.  d_temperature, d_top_p: [B] fp32; d_top_k: [B] int32 (<= 0 or >= V:
 * no top-k; top_p >= 1: no top-p).  A sequence with T_b not > 0 and finite
 * or top_p_b not > 0 gets ST_BADPARAM.  Workspace:
 * spec_verify_sampling_workspace_bytes(B, K, V) bytes, 256-byte aligned, its
 * first 256 bytes zeroed once by spec_verify_workspace_init; the rest holds
 * the cuts of the call.  dbg as spec_verify (row_z sums the kept tokens; q_d
 * is not written).  V limits as spec_verify's one-hot case.  The cut and the
 * verification: two launches (three with bf16 targets). */
size_t spec_verify_sampling_workspace_bytes(int32_t B, int32_t K, int32_t V);
int spec_verify_sampling(const void* d_target, int32_t target_dtype, const int32_t* d_draft,
                         const int32_t* d_draft_len, int32_t B, int32_t K, int32_t V,
                         const float* d_temperature, const int32_t* d_top_k,
                         const float* d_top_p, uint64_t seed, uint64_t step,
                         int32_t* d_accept_len, int32_t* d_out_token, int32_t* d_emit,
                         int32_t* d_emit_len, int32_t* d_status, const spec_verify_debug* dbg,
                         void* d_workspace, size_t ws_bytes, samspec_stream_t stream);

/* One decode step of model-free speculative decoding ([P1] §1.1: verify, then
 * update each sequence's D-SAM with the verified tokens, then draft; [P1]
 * §3.1.1: whether a step speculates at all is the caller's choice of K and
 * K_next, e.g. only while the number of active sequences is at most a
 * threshold):
 *   1. spec_verify of n sequences (one-hot drafts: logits [n, K+1, V],
 *      d_draft [n, K] with d_draft_len [n] or NULL; K = 0 verifies the bonus
 *      row only, i.e. plain decoding) into accept_len / out_token / status
 *      and the required d_emit [n, K+1] / d_emit_len [n];
 *   2. sam_step_rows: automaton d_rows[i] (or i) is extended by its emitted
 *      tokens (none for a sequence with a non-zero status) and drafts K_next
 *      tokens into d_next_draft [n, K_next] / d_next_draft_len [n] (all 0
 *      when K_next = 0; d_next_draft may then be NULL).
 * d_next_draft may alias d_draft (the verification has read it by then).
 * Two launches on `stream`; workspace as for spec_verify.  Errors as for the
 * two calls. */
int sam_spec_step(sam_batch* batch, const int32_t* d_rows, int32_t n, const void* d_target,
                  int32_t target_dtype, const int32_t* d_draft, const int32_t* d_draft_len,
                  int32_t K, int32_t V, float temperature, uint64_t seed, uint64_t step,
                  int32_t* d_accept_len, int32_t* d_out_token, int32_t* d_emit,
                  int32_t* d_emit_len, int32_t* d_status, const spec_verify_debug* dbg,
                  int32_t K_next, int32_t* d_next_draft, int32_t* d_next_draft_len,
                  int32_t* d_match_len, int32_t* d_min_endpos, void* d_workspace,
                  size_t ws_bytes, samspec_stream_t stream);

/* Test hook of the verification kernels' bounded waits.  Every on-chip wait of
 * spec_verify, spec_verify_noalloc, spec_verify_tree, spec_verify_sampling and
 * sam_spec_step's verification (a staging buffer to fill or to free, the
 * records of a tile, an idle sequence slot) gives up after `ns` nanoseconds of
 * global time instead of the default 2 s; ns = 0 restores the default.  A
 * kernel whose wait runs out marks every sequence it has not finished with
 * ST_TIMEOUT (accept_len and out_token -1, emit_len 0), waits for its own
 * copies in flight to land (up to 2 s, a limit this hook does not shorten)
 * and returns; sequences it finished keep their results, and the context and
 * the workspace stay usable.  Process-wide; applies to launches made after
 * the call (a launch captured in a CUDA graph keeps the value in force at its
 * capture).  Returns the previous limit.  Meant for tests of the timeout
 * path: production code never needs it. */
uint64_t samspec_set_wait_limit_ns(uint64_t ns);

/* Philox4x32-10 uniforms exactly as spec_verify draws them, for inspection:
 * d_u[2 * (b * (K+1) + j) + {0,1}] = (u_j, u'_j) of sequence b, for
 * 0 <= b < B and 0 <= j <= K ([B, K+1, 2] fp32, device).  Asynchronous. */
int spec_uniforms(int32_t B, int32_t K, uint64_t seed, uint64_t step, float* d_u,
                  samspec_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SAMSPEC_H_ */
