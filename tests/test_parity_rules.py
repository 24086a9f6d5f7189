"""The parity rules reject planted device errors (no GPU).

The GPU parity tests pass a device result and the oracle's result on the
same inputs to the comparison helpers in tests/parity.py.  Here the oracle's
own result stands in for the device's, first unchanged (it must pass with
nothing excused), then with one planted error each: a wrong emitted token, a
wrong accept length, a wrong status, a probability off by 1e-5 relative, a
wrong greedy argmax, a wrong top-k/top-p cut, a wrong tree path.  Every
planted error must fail the comparison.  One case builds a genuine tie
(a coin within rounding of its accept threshold): the other decision there
is excused, and counts against the 1e-4 budget.
"""
import copy

import numpy as np
import pytest

import oracle
from parity import compare_sampling, compare_trees, compare_verify

SEED, STEP = 5, 3


def _linear_case(T, B=64, K=3, V=512):
    rng = np.random.default_rng(11)
    target = rng.normal(0.0, 2.0, (B, K + 1, V)).astype(np.float32)
    # drafts from each row's five largest logits, so that some are accepted
    top = np.argsort(-target[:, :K, :], axis=2)[:, :, :5]
    pick = rng.integers(0, 5, (B, K))
    draft = np.take_along_axis(top, pick[:, :, None], axis=2)[:, :, 0].astype(np.int32)
    o = oracle.verify(target, draft, temperature=T, seed=SEED, step=STEP)
    return target, draft, o


def _cmp(g, o, target, draft, T, **kw):
    return compare_verify(g, o, lambda b: target[b], draft, None, T, **kw)


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_unchanged_result_passes(T):
    target, draft, o = _linear_case(T)
    d, e = _cmp(copy.deepcopy(o), o, target, draft, T)
    assert e == 0 and d > 64
    assert 0 < int((o["accept_len"] > 0).sum()) < 64  # both outcomes present


def _first(cond):
    idx = np.flatnonzero(cond)
    assert idx.size, "the case lacks the sequence a plant needs"
    return int(idx[0])


@pytest.mark.parametrize("T", [1.0, 0.0])
@pytest.mark.parametrize("plant", ["token", "longer", "shorter", "status"])
def test_wrong_decisions_fail(T, plant):
    target, draft, o = _linear_case(T)
    K, V = draft.shape[1], target.shape[2]
    g = copy.deepcopy(o)
    if plant == "token":
        b = _first(o["status"] == 0)
        g["out_token"][b] = (o["out_token"][b] + V // 2) % V
    elif plant == "longer":
        b = _first(o["accept_len"] < K)
        g["accept_len"][b] += 1
    elif plant == "shorter":
        b = _first(o["accept_len"] > 0)
        g["accept_len"][b] -= 1
    else:
        b = 0
        g["status"][b] = oracle.BADROW
    with pytest.raises(AssertionError):
        _cmp(g, o, target, draft, T)


@pytest.mark.parametrize("key", ["row_z", "row_m", "p_d", "q_d"])
def test_statistics_off_by_1e5_fail(key):
    target, draft, o = _linear_case(1.0)
    b = _first(o["accept_len"] > 0)
    g = copy.deepcopy(o)
    g[key][b, 0] *= 1 + 1e-7  # inside the 1e-6 relative tolerance
    _cmp(g, o, target, draft, 1.0)
    g[key][b, 0] *= 1 + 1e-5
    with pytest.raises(AssertionError):
        _cmp(g, o, target, draft, 1.0)


def test_greedy_argmax_must_match_exactly():
    target, draft, o = _linear_case(0.0)
    g = copy.deepcopy(o)
    g["row_arg"][0, 0] = (o["row_arg"][0, 0] + 1) % target.shape[2]
    with pytest.raises(AssertionError):
        _cmp(g, o, target, draft, 0.0)


def test_a_genuine_tie_is_excused_and_counted():
    # one sequence, one draft d = 0 over V = 2: choose the logit so that
    # p(d) = softmax([a, 0])[0] equals the accept coin u up to fp32 rounding
    u, _ = oracle.uniforms(SEED, STEP, 0, 0)
    a = np.float32(np.log(u / (1.0 - u)))
    target = np.array([[[a, 0.0], [0.3, -0.2]]], np.float32)
    draft = np.zeros((1, 1), np.int32)
    o = oracle.verify(target, draft, temperature=1.0, seed=SEED, step=STEP)
    assert abs(o["u_acc"][0, 0] - o["p_d"][0, 0]) < 1e-6
    g = copy.deepcopy(o)
    g["accept_len"][0] = 1 - o["accept_len"][0]  # the other decision
    d, e = _cmp(g, o, target, draft, 1.0, check_probs=False, budget=False)
    assert e == 1
    with pytest.raises(AssertionError):  # 1 excused of 3 decisions is over 1e-4
        _cmp(g, o, target, draft, 1.0, check_probs=False)


# ---- per-request truncation --------------------------------------------------

def _sampling_case(B=48, K=2, V=256):
    rng = np.random.default_rng(23)
    rows = rng.normal(0.0, 2.0, (B, K + 1, V)).astype(np.float32)
    top = np.argsort(-rows[:, :K, :], axis=2)[:, :, :4]
    pick = rng.integers(0, 4, (B, K))
    draft = np.take_along_axis(top, pick[:, :, None], axis=2)[:, :, 0].astype(np.int32)
    T = rng.choice(np.array([0.6, 0.8, 1.0]), B)
    k = rng.choice(np.array([0, 20, 50], np.int32), B)
    p = rng.choice(np.array([0.9, 0.95, 1.0]), B)
    o = oracle.verify_sampling(rows, draft, temperature=T, top_k=k, top_p=p, seed=SEED, step=STEP)
    return rows, draft, T, k, p, o


def _cmp_s(g, tau_g, case):
    rows, draft, T, k, p, o = case
    return compare_sampling(g, o, rows, draft, T, k, p, tau_g)


def test_sampling_unchanged_passes():
    case = _sampling_case()
    o = case[-1]
    assert np.all(o["status"] == 0)
    d, e = _cmp_s(copy.deepcopy(o), o["tau"].copy(), case)
    assert e == 0 and d > 0


@pytest.mark.parametrize("plant", ["token", "token_outside_cut", "accept_len", "cut_topk", "cut_topp"])
def test_sampling_wrong_results_fail(plant):
    case = _sampling_case()
    rows, draft, T, k, p, o = case
    V = rows.shape[2]
    g, tau_g = copy.deepcopy(o), o["tau"].copy()
    if plant in ("token", "token_outside_cut"):
        b = _first((k > 0) | (p < 1))
        L = int(o["accept_len"][b])
        kept = np.flatnonzero(rows[b, L] >= tau_g[b, L])
        cut = np.flatnonzero(rows[b, L] < tau_g[b, L])
        if plant == "token":  # another kept token, far from the coin's interval
            others = kept[kept != o["out_token"][b]]
            g["out_token"][b] = int(others[len(others) // 2])
        else:
            g["out_token"][b] = int(cut[0])
    elif plant == "accept_len":
        b = _first(o["accept_len"] < draft.shape[1])
        g["accept_len"][b] += 1
    else:
        # keep one more token: move row 0's cut down to the next smaller logit,
        # in a sequence cut by top-k alone, or by top-p alone; the emitted
        # token differs too, since cuts are compared where decisions differ
        sel = (k > 0) & (p >= 1) if plant == "cut_topk" else (k == 0) & (p < 1)
        b = _first(sel)
        x = np.unique(rows[b, 0])
        tau_g[b, 0] = x[int(np.searchsorted(x, tau_g[b, 0])) - 1]
        L = int(o["accept_len"][b])
        kept = np.flatnonzero(rows[b, L] >= o["tau"][b, L])
        g["out_token"][b] = int(kept[kept != o["out_token"][b]][0])
        with pytest.raises(AssertionError, match=rf"^\({b}, 0\)$"):  # the cut rule itself
            _cmp_s(g, tau_g, case)
        return
    with pytest.raises(AssertionError):
        _cmp_s(g, tau_g, case)


# ---- draft trees --------------------------------------------------------------

def _tree_case(T, B=32, N=8, V=64):
    rng = np.random.default_rng(31)
    rows = rng.normal(0.0, 1.5, (B, N, V)).astype(np.float32)
    tok = np.full((B, N), -1, np.int32)
    fc = np.full((B, N), -1, np.int32)
    ns = np.full((B, N), -1, np.int32)
    for b in range(B):
        parent_of = [-1]
        last_child = {}
        for n in range(1, N):
            par = int(rng.integers(0, n))
            parent_of.append(par)
            used = {int(tok[b, c]) for c in range(1, n) if parent_of[c] == par}
            # children drawn from the parent row's largest logits
            order = [int(t) for t in np.argsort(-rows[b, par]) if int(t) not in used]
            tok[b, n] = order[int(rng.integers(0, 3))]
            if par in last_child:
                ns[b, last_child[par]] = n
            else:
                fc[b, par] = n
            last_child[par] = n
    o = oracle.tree_verify(rows, tok, fc, ns, temperature=T, seed=SEED, step=STEP)
    o["emit"] = np.full((B, N + 1), -1, np.int32)
    for b in range(B):
        L = int(o["accept_len"][b])
        o["emit"][b, :L + 1] = [int(tok[b, n]) for n in o["path"][b, :L]] + [int(o["out_token"][b])]
    return rows, tok, fc, ns, o


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_tree_unchanged_passes(T):
    rows, tok, fc, ns, o = _tree_case(T)
    assert np.all(o["status"] == 0) and np.any(o["accept_len"] > 0)
    d, e = compare_trees(copy.deepcopy(o), o, rows, tok, fc, ns, T, SEED, STEP)
    assert e == 0


@pytest.mark.parametrize("T", [1.0, 0.0])
@pytest.mark.parametrize("plant", ["token", "path", "emit"])
def test_tree_wrong_results_fail(T, plant):
    rows, tok, fc, ns, o = _tree_case(T)
    V = rows.shape[2]
    g = copy.deepcopy(o)
    if plant == "token":
        b = 0
        g["out_token"][b] = (o["out_token"][b] + V // 2) % V
    elif plant == "path":
        b = _first(o["accept_len"] > 0)
        g["accept_len"][b] -= 1
        g["path"][b, int(g["accept_len"][b])] = -1
    else:
        b = _first(o["accept_len"] > 0)
        g["emit"][b, 0] = (g["emit"][b, 0] + 1) % V
    with pytest.raises(AssertionError):
        compare_trees(g, o, rows, tok, fc, ns, T, SEED, STEP)
