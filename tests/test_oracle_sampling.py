"""Pins of the oracle's per-request sampling parameters (gogongxt.com notes
"投机采样", SGLang 的实现: per-request temperature, top-k renormalisation and
top-p renormalisation of the target probabilities before the drafts are
tested), each checked by a route other than the oracle's own:
  * the kept sets by brute force on tiny rows with ties: top-k keeps a token
    iff fewer than k tokens have a strictly larger logit; top-p keeps a
    token iff the renormalised mass strictly above it is below top_p (a
    double loop), and the kept set is the smallest such top set;
  * disabled truncation (k <= 0 or >= V, top_p >= 1) is the plain
    verification; top_k = 1 is greedy verification at any temperature;
  * a power-of-two temperature equals the same logits scaled at T = 1;
  * the emitted first token follows the truncated distribution (chi-square);
  * bad parameters are refused per sequence."""
import numpy as np
import pytest
from scipy import stats

import oracle
import workloads


def _brute(row, T, k, top_p):
    x = row.astype(np.float64)
    V = len(x)
    p = np.exp(x / T - (x / T).max())
    p /= p.sum()
    keep = np.ones(V, bool)
    if 0 < k < V:
        keep = np.array([sum(x[u] > x[v] for u in range(V)) < k for v in range(V)])
    pk = np.where(keep, p, 0.0)
    pk /= pk.sum()
    if top_p < 1.0:
        keep2 = np.array([keep[v] and sum(pk[u] for u in range(V) if x[u] > x[v]) < top_p
                          for v in range(V)])
        keep = keep2
    pp = np.where(keep, p, 0.0)
    return pp / pp.sum(), keep


@pytest.mark.parametrize("V", [2, 5, 8])
def test_kept_sets_by_brute_force(V):
    rng = np.random.default_rng(V)
    for trial in range(300):
        row = rng.integers(-3, 4, V).astype(np.float32) * 0.5  # few distinct values: ties
        T = float(rng.choice([0.5, 1.0, 1.7]))
        k = int(rng.integers(-1, V + 2))
        top_p = float(rng.choice([0.3, 0.5, 0.8, 0.95, 1.0, 1.5]))
        pp, tau = oracle.truncate_row(row, T, k, top_p)
        want, keep = _brute(row, T, k, top_p)
        np.testing.assert_allclose(pp, want, rtol=1e-12, atol=1e-15)
        assert tau == row[keep].min()
        # the smallest top set reaching top_p: dropping its lowest logit group
        # leaves less than top_p of the top-k mass
        if top_p < 1.0:
            pk, kk = _brute(row, T, k, 1.0)
            assert pk[keep].sum() >= top_p - 1e-12
            lower = keep & (row > row[keep].min())
            assert pk[lower].sum() < top_p


def test_disabled_truncation_is_plain_verification():
    rng = np.random.default_rng(1)
    B, K, V = 64, 3, 300
    logits = workloads.gaussian_logits(rng, (B, K + 1, V), 2.0)
    draft = np.argsort(-logits[:, :K], axis=-1)[..., 1].astype(np.int32)
    plain = oracle.verify(logits, draft, None, temperature=0.8, seed=4, step=2)
    for k, p in ((0, 1.0), (V, 1.0), (-1, 2.0)):
        s = oracle.verify_sampling(logits, draft, None, 0.8, k, p, seed=4, step=2)
        np.testing.assert_array_equal(s["accept_len"], plain["accept_len"])
        np.testing.assert_array_equal(s["out_token"], plain["out_token"])


def test_top1_is_greedy_at_any_temperature():
    rng = np.random.default_rng(2)
    B, K, V = 64, 4, 200
    logits = workloads.gaussian_logits(rng, (B, K + 1, V), 2.0)
    am = np.argmax(logits[:, :K], axis=-1).astype(np.int32)
    draft = np.where(rng.random((B, K)) < 0.7, am, (am + 1) % V).astype(np.int32)
    greedy = oracle.verify(logits, draft, None, temperature=0.0)
    for T in (0.3, 1.0, 4.0):
        s = oracle.verify_sampling(logits, draft, None, T, 1, 1.0, seed=9, step=int(10 * T))
        np.testing.assert_array_equal(s["accept_len"], greedy["accept_len"])
        np.testing.assert_array_equal(s["out_token"], greedy["out_token"])


def test_temperature_scales_the_logits():
    rng = np.random.default_rng(3)
    row = workloads.gaussian_logits(rng, (400,), 2.0)
    for k, p in ((10, 1.0), (0, 0.9), (50, 0.7)):
        a, ta = oracle.truncate_row(row, 2.0, k, p)
        b, tb = oracle.truncate_row(row / 2.0, 1.0, k, p)
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-300)
        assert tb == ta / 2.0


def test_first_token_follows_the_truncated_distribution():
    rng = np.random.default_rng(5)
    V, B, T, k, p = 12, 200000, 0.8, 7, 0.9
    row = workloads.gaussian_logits(rng, (V,), 1.0)
    logits = np.broadcast_to(np.stack([row, row]), (B, 2, V)).copy()
    draft = np.full((B, 1), int(np.argsort(-row)[2]), np.int32)
    s = oracle.verify_sampling(logits, draft, None, T, k, p, seed=13, step=0)
    assert (s["status"] == 0).all()
    first = np.where(s["accept_len"] >= 1, draft[:, 0], s["out_token"])
    want, keep = _brute(row, T, k, p)
    counts = np.bincount(first, minlength=V)
    assert (counts[~keep] == 0).all()
    res = stats.chisquare(counts[keep], want[keep] * B)
    assert res.pvalue > 1e-3, res


def test_bad_parameters_are_refused():
    rng = np.random.default_rng(6)
    B, K, V = 6, 2, 50
    logits = workloads.gaussian_logits(rng, (B, K + 1, V), 1.0)
    draft = np.zeros((B, K), np.int32)
    T = np.array([0.0, np.inf, np.nan, 1.0, 1.0, 1.0])
    p = np.array([0.9, 0.9, 0.9, 0.0, np.nan, 0.9])
    s = oracle.verify_sampling(logits, draft, None, T, 5, p)
    assert list(s["status"]) == [8, 8, 8, 8, 8, 0]
    assert (s["accept_len"][:5] == -1).all()


def test_signed_zeros_are_one_value():
    """+0 and -0 compare equal, so a row mixing them truncates exactly as the
    row with every zero positive (ties at a cut are kept on both sides of the
    sign), checked against the brute-force definition."""
    row = np.zeros(9, np.float32)
    row[:4] = -0.0
    row[[6, 8]] = [1.5, 0.75]
    pos = np.abs(row)
    for T, k, top_p in ((1.0, 3, 1.0), (1.0, 0, 0.6), (0.7, 5, 0.9), (1.3, 2, 0.99)):
        pa, ta = oracle.truncate_row(row, T, k, top_p)
        pb, tb = oracle.truncate_row(pos, T, k, top_p)
        np.testing.assert_array_equal(pa, pb)
        assert ta == tb
        pbr, keep = _brute(pos, T, k, top_p)
        np.testing.assert_allclose(pa, pbr, rtol=1e-12, atol=0)
        assert ta == pos[keep].min()


def test_negative_infinity_logits():
    """-inf logits have zero probability: top-k still counts them (a k beyond
    the finite logits cuts at -inf and keeps every finite one), and top-p
    never needs them."""
    row = np.array([2.0, -np.inf, 0.5, -np.inf, 1.0, -np.inf], np.float32)
    p, tau = oracle.truncate_row(row, 1.0, 5, 1.0)
    assert tau == -np.inf
    assert (p[np.isfinite(row)] > 0).all() and (p[~np.isfinite(row)] == 0).all()
    np.testing.assert_allclose(p.sum(), 1.0, rtol=1e-15)
    p, tau = oracle.truncate_row(row, 1.0, 0, 0.999999)
    assert tau == 0.5 and (p[~np.isfinite(row)] == 0).all()
    p, tau = oracle.truncate_row(row, 1.0, 2, 1.0)
    assert tau == 1.0 and np.count_nonzero(p) == 2


def test_constant_row_keeps_everything():
    """Every logit equal: any top-k keeps all of them (ties at the k-th), any
    top-p keeps all of them (nothing lies strictly above), and the result is
    uniform."""
    row = np.full(7, 0.25, np.float32)
    for k, top_p in ((1, 1.0), (3, 0.5), (0, 0.01), (6, 0.99)):
        p, tau = oracle.truncate_row(row, 0.8, k, top_p)
        assert tau == np.float32(0.25)
        np.testing.assert_allclose(p, np.full(7, 1 / 7), rtol=1e-14)
