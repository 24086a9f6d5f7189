"""Pins of the oracle's verification against what the pages and the mathematics
fix (no GPU):

* greedy verification (gogongxt "投机采样" notes, 贪婪采样) equals numpy's argmax
  (lowest index on ties) row by row, and the accepted length is a direct
  prefix comparison;
* the temperature softmax (same notes, SGLang 的实现) equals scipy's softmax and
  logsumexp;
* rejection sampling (nxbn.cn article §2.2; CANN SAM article §1.1) makes every
  emitted token follow the target distribution, whatever the drafts: a
  chi-square test per output position, and the acceptance frequency matches
  sum_v min(p_v, q_v) (one-hot drafts: p(d));
* end-to-end: SAM drafting + verification of a toy target decodes exactly the
  plain greedy sequence, and in sampling mode its short continuations follow
  direct sampling;
* malformed rows and drafts are reported, not sampled.
"""
import numpy as np
import pytest
from scipy import special, stats

import oracle
import workloads


def test_greedy_equals_argmax_and_prefix():
    rng = np.random.default_rng(21)
    B, K, V = 64, 5, 97
    logits = workloads.gaussian_logits(rng, (B, K + 1, V), 1.0)
    amax = np.argmax(logits, axis=-1)
    draft = amax[:, :K].copy()
    # corrupt a random position per sequence (or none)
    cut = rng.integers(0, K + 1, size=B)
    for b in range(B):
        if cut[b] < K:
            draft[b, cut[b]] = (draft[b, cut[b]] + 1 + rng.integers(0, V - 1)) % V
    dl = rng.integers(0, K + 1, size=B).astype(np.int32)
    r = oracle.verify(logits, draft, dl, temperature=0.0)
    for b in range(B):
        L = 0
        while L < dl[b] and draft[b, L] == amax[b, L]:
            L += 1
        assert r["accept_len"][b] == L
        assert r["out_token"][b] == amax[b, L]
        assert r["status"][b] == oracle.OK


def test_greedy_ties_take_lowest_index():
    V = 16
    logits = np.zeros((1, 2, V), np.float32)
    logits[0, 0, [3, 7, 11]] = 5.0
    logits[0, 1, [2, 9]] = 1.0
    r = oracle.verify(logits, np.array([[3]]), temperature=0.0)
    assert r["accept_len"][0] == 1 and r["out_token"][0] == 2
    r = oracle.verify(logits, np.array([[7]]), temperature=0.0)
    assert r["accept_len"][0] == 0 and r["out_token"][0] == 3
    assert np.argmax(logits[0, 0]) == 3


@pytest.mark.parametrize("T", [0.3, 0.7, 1.0, 2.5])
def test_softmax_matches_scipy(T):
    rng = np.random.default_rng(22)
    B, K, V = 8, 3, 1000
    logits = workloads.gaussian_logits(rng, (B, K + 1, V), 2.0)
    draft = rng.integers(0, V, size=(B, K)).astype(np.int32)
    r = oracle.verify(logits, draft, temperature=T, seed=5, step=9)
    for b in range(B):
        for j in range(r["accept_len"][b] + 1):
            x = logits[b, j].astype(np.float64) / T
            assert abs(r["row_m"][b, j] - x.max()) <= 1e-15 * abs(x.max())
            lse = special.logsumexp(x)
            assert abs(np.log(r["row_z"][b, j]) + r["row_m"][b, j] - lse) <= 1e-12 * max(1, abs(lse))
            if j < r["accept_len"][b] + 1 and j < K and not np.isnan(r["p_d"][b, j]):
                p = special.softmax(x)
                assert abs(r["p_d"][b, j] - p[draft[b, j]]) <= 1e-12 * p[draft[b, j]]


def _tiny_case(rng, V, K, T, with_draft):
    target = workloads.gaussian_logits(rng, (K + 1, V), 1.5)
    p = special.softmax(target.astype(np.float64) / T, axis=-1)
    if with_draft:
        draftl = (target[:K] + workloads.gaussian_logits(rng, (K, V), 1.0)).astype(np.float32)
        q = special.softmax(draftl.astype(np.float64) / T, axis=-1)
    else:
        draftl, q = None, None
    return target, draftl, p, q


@pytest.mark.parametrize("with_draft", [False, True])
def test_rejection_sampling_is_lossless_chi_square(with_draft):
    """Each emitted position follows the target distribution p_j."""
    rng = np.random.default_rng(23 + with_draft)
    V, K, T = 8, 3, 0.8
    target, draftl, p, q = _tiny_case(rng, V, K, T, with_draft)
    B, steps = 100000, 10
    tgt = np.broadcast_to(target, (B, K + 1, V))
    dlg = None if draftl is None else np.broadcast_to(draftl, (B, K, V))
    emitted = [[] for _ in range(K + 1)]
    acc_hits = np.zeros(K)
    acc_tries = np.zeros(K)
    for step in range(steps):
        if with_draft:
            # drafts sampled from q_j (inverse CDF with a separate generator)
            u = rng.random((B, K))
            draft = np.stack([np.searchsorted(np.cumsum(q[j]), u[:, j], side="right")
                              for j in range(K)], axis=1).clip(0, V - 1).astype(np.int32)
        else:
            draft = np.tile(np.array([[1, 6, 3]], np.int32), (B, 1))
        r = oracle.verify(tgt, draft, temperature=T, seed=1234, step=step, draft_logits=dlg)
        L, out = r["accept_len"], r["out_token"]
        for j in range(K + 1):
            reach = L >= j
            tok = np.where(L[reach] > j, draft[reach, min(j, K - 1)], out[reach])
            emitted[j].append(tok)
        for j in range(K):
            tried = L >= j
            acc_tries[j] += tried.sum()
            acc_hits[j] += (L[tried] > j).sum()
    n_tests = 2 * K + 1
    for j in range(K + 1):
        tok = np.concatenate(emitted[j])
        hist = np.bincount(tok, minlength=V)
        pval = stats.chisquare(hist, p[j] * hist.sum()).pvalue
        assert pval > 1e-3 / n_tests, (j, pval)
    for j in range(K):
        want = np.minimum(p[j], q[j]).sum() if with_draft else p[j][[1, 6, 3][j]]
        n = acc_tries[j]
        z = (acc_hits[j] - n * want) / np.sqrt(n * want * (1 - want))
        assert abs(z) < stats.norm.isf(1e-3 / n_tests / 2), (j, z)


def test_bonus_row_samples_target():
    rng = np.random.default_rng(25)
    V, K, T = 6, 2, 1.3
    target = workloads.gaussian_logits(rng, (K + 1, V), 1.0)
    p0 = special.softmax(target[0].astype(np.float64) / T)
    B = 200000
    r = oracle.verify(np.broadcast_to(target, (B, K + 1, V)), np.zeros((B, K), np.int32),
                      np.zeros(B, np.int32), temperature=T, seed=3, step=1)
    assert np.all(r["accept_len"] == 0)
    hist = np.bincount(r["out_token"], minlength=V)
    assert stats.chisquare(hist, p0 * B).pvalue > 1e-3


def test_a_subset_with_its_sequence_indices_equals_the_full_batch():
    # a sequence's coins are keyed by its index (counter word 1), so a subset
    # verified with the caller's indices gives the full batch's results for
    # those sequences, and its resample coins are U(word 1) of those indices
    rng = np.random.default_rng(27)
    B, K, V, T = 12, 3, 200, 1.0
    target = workloads.gaussian_logits(rng, (B, K + 1, V), 2.0)
    top = np.argsort(-target[:, :K], axis=2)[:, :, :5]
    draft = np.take_along_axis(top, rng.integers(0, 5, (B, K, 1)), axis=2)[:, :, 0].astype(np.int32)
    full = oracle.verify(target, draft, temperature=T, seed=4, step=6)
    idx = np.array([7, 2, 11, 5])
    sub = oracle.verify(target[idx], draft[idx], temperature=T, seed=4, step=6, seq_index=idx)
    for key in ("accept_len", "out_token", "status", "u_res"):
        assert np.array_equal(sub[key], full[key][idx]), key
    for i, b in enumerate(idx):
        assert sub["u_res"][i] == oracle.uniforms(4, 6, int(b), int(sub["accept_len"][i]))[1]
    plain = oracle.verify(target[idx], draft[idx], temperature=T, seed=4, step=6)
    assert not np.array_equal(plain["u_res"], sub["u_res"])


@pytest.mark.parametrize("T", [1.0, 0.7])
def test_resample_lies_in_its_cdf_interval(T):
    # at T != 1 too: the draft distribution is softmax(draft logits / T)
    rng = np.random.default_rng(26)
    B, K, V = 16, 3, 300
    target = workloads.gaussian_logits(rng, (B, K + 1, V), 2.0)
    draftl = (target[:, :K] + workloads.gaussian_logits(rng, (B, K, V), 1.0)).astype(np.float32)
    draft = rng.integers(0, V, size=(B, K)).astype(np.int32)
    for dlg in (None, draftl):
        r = oracle.verify(target, draft, temperature=T, seed=8, step=2, draft_logits=dlg)
        for b in range(B):
            L = r["accept_len"][b]
            rej = draft[b, L] if L < K else -1
            lo, hi, mass = oracle.cdf_interval(target[b, L], T, rej, r["out_token"][b],
                                               None if (dlg is None or L == K) else dlg[b, L])
            assert lo <= r["u_res"][b] < hi
            assert abs(mass - r["res_mass"][b]) <= 1e-12
            u_acc, u_res = oracle.uniforms(8, 2, b, L)
            assert u_res == r["u_res"][b]


def test_malformed_rows_and_drafts():
    V, K = 8, 2
    base = np.zeros((1, K + 1, V), np.float32)
    d = np.array([[1, 2]], np.int32)
    x = base.copy(); x[0, 0, 3] = np.nan
    assert oracle.verify(x, d, temperature=0.0)["status"][0] == oracle.BADROW
    assert oracle.verify(x, d, temperature=1.0)["status"][0] == oracle.BADROW
    x = base.copy(); x[0, 0, :] = -np.inf
    assert oracle.verify(x, d, temperature=0.0)["status"][0] == oracle.BADROW
    assert oracle.verify(x, d, temperature=1.0)["status"][0] == oracle.BADROW
    x = base.copy(); x[0, 0, 5] = np.inf
    assert oracle.verify(x, d, temperature=1.0)["status"][0] == oracle.BADROW
    r = oracle.verify(x, np.array([[5, 2]], np.int32), temperature=0.0)
    assert r["status"][0] == oracle.OK and r["accept_len"][0] >= 1
    x = base.copy(); x[0, 0, :4] = -np.inf  # masked vocabulary is fine
    assert oracle.verify(x, d, temperature=1.0)["status"][0] == oracle.OK
    assert oracle.verify(base, np.array([[1, 8]], np.int32), temperature=1.0)["status"][0] == oracle.BADDRAFT
    assert oracle.verify(base, d, np.array([3], np.int32), temperature=1.0)["status"][0] == oracle.BADDRAFT
    # draft_len bounds which tokens are checked
    assert oracle.verify(base, np.array([[1, 99]], np.int32), np.array([1], np.int32),
                         temperature=1.0)["status"][0] == oracle.OK


# ---------------------------------------------------------------------------
# End-to-end losslessness with a toy target model.
# ---------------------------------------------------------------------------

def _toy_logits(prefix, V, ctx=3, seed=99):
    """Logits of a toy target: a seeded function of the last `ctx` tokens, so
    that the generated text repeats and the automaton's drafts get accepted."""
    key = (seed,) + tuple(int(t) for t in prefix[-ctx:])
    rng = np.random.default_rng(abs(hash(key)) % (2**63))
    return (rng.standard_normal(V) * 3.0).astype(np.float32)


def _spec_decode(prompt, n_out, V, K, T, seed):
    sam = oracle.Sam(V)
    sam.extend(prompt)
    text = list(prompt)
    step = 0
    while len(text) - len(prompt) < n_out:
        draft, dl, _, _ = sam.draft(K)
        rows = np.stack([_toy_logits(text + list(draft[:j]), V) for j in range(K + 1)])
        r = oracle.verify(rows[None], draft[None].clip(0), np.array([dl], np.int32),
                          temperature=T, seed=seed, step=step)
        L = int(r["accept_len"][0])
        new = list(draft[:L]) + [int(r["out_token"][0])]
        text += new
        sam.extend(new)
        step += 1
    return text[len(prompt):len(prompt) + n_out], step


def test_end_to_end_greedy_equals_plain_decoding():
    V, K = 16, 4
    rng = np.random.default_rng(31)
    for trial in range(4):
        prompt = list(rng.integers(0, V, size=20))
        plain = []
        text = list(prompt)
        for _ in range(120):
            t = int(np.argmax(_toy_logits(text, V)))
            plain.append(t)
            text.append(t)
        spec, steps = _spec_decode(prompt, 120, V, K, 0.0, 0)
        assert spec == plain
        assert steps < 120  # drafts were accepted along the way


def test_end_to_end_sampling_matches_direct_sampling():
    V, K, T = 4, 3, 1.0
    prompt = [0, 1, 2, 3, 0, 1]
    counts = np.zeros((V, V))
    n = 4000
    for s in range(n):
        out, _ = _spec_decode(prompt, 2, V, K, T, seed=1000 + s)
        counts[out[0], out[1]] += 1
    p0 = special.softmax(_toy_logits(prompt, V).astype(np.float64) / T)
    want = np.array([[p0[a] * special.softmax(_toy_logits(prompt + [a], V).astype(np.float64) / T)[c]
                      for c in range(V)] for a in range(V)])
    assert stats.chisquare(counts.ravel(), want.ravel() * n).pvalue > 1e-3
