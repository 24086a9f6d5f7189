"""Comparison helpers for the GPU-vs-oracle parity tests (no method arithmetic:
only the comparison rules).

Verification decisions must be identical, except where a coin lies within
1e-6 of the oracle's threshold p/q (accept test) or of a boundary of the
oracle's CDF interval of the GPU's token (resample); such excused mismatches
must be at most 1e-4 of all decisions.  Probabilities must agree within 1e-6
relative.
"""
from __future__ import annotations

import numpy as np

import oracle

BAND = 1e-6
PROB_RTOL = 1e-6


def rel_err(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return np.abs(a - b) / np.maximum(np.abs(b), 1e-300)


def compare_verify(g, o, target_rows, draft, draft_len, T, draft_rows=None, check_probs=True,
                   budget=True):
    """g: dict of numpy arrays from the GPU; o: oracle.verify output on the
    same inputs.  target_rows(b) -> [K+1, V] float32 rows of sequence b,
    draft_rows(b) -> [K, V] or None.  Returns (decisions, excused).  With
    budget=False the 1e-4 share is left to the caller (counted over many
    calls)."""
    B, K1 = o["row_m"].shape
    K = K1 - 1
    decisions = 0
    excused = 0
    for b in range(B):
        assert g["status"][b] == o["status"][b], (b, g["status"][b], o["status"][b])
        if o["status"][b] != 0:
            assert g["accept_len"][b] == -1 and g["out_token"][b] == -1
            continue
        Lg, Lo = int(g["accept_len"][b]), int(o["accept_len"][b])
        nb = K if draft_len is None else int(draft_len[b])
        decisions += min(Lg, Lo) + 1 + 1
        if Lg != Lo:
            j = min(Lg, Lo)
            assert T > 0, f"greedy accept length differs at b={b}: gpu {Lg} oracle {Lo}"
            u = o["u_acc"][b, j]
            thr = o["p_d"][b, j] / o["q_d"][b, j]
            assert abs(u - thr) < BAND, f"b={b} j={j}: u={u} threshold={thr} (gpu L={Lg}, oracle L={Lo})"
            excused += 1
            continue
        if g["out_token"][b] != o["out_token"][b]:
            assert T > 0, f"greedy token differs at b={b}"
            L = Lo
            rej = int(draft[b, L]) if L < nb else -1
            drow = None
            if draft_rows is not None and L < nb:
                drow = draft_rows(b)[L]
            lo, hi, _ = oracle.cdf_interval(target_rows(b)[L], T, rej, int(g["out_token"][b]), drow)
            u = o["u_res"][b]
            assert lo - BAND <= u < hi + BAND, f"b={b}: u'={u} outside [{lo}, {hi}) of gpu token"
            excused += 1
        if check_probs:
            for j in range(Lo + 1):
                if T > 0:
                    assert rel_err(g["row_m"][b, j], o["row_m"][b, j]) < PROB_RTOL, (b, j)
                    assert rel_err(g["row_z"][b, j], o["row_z"][b, j]) < PROB_RTOL, (b, j, g["row_z"][b, j], o["row_z"][b, j])
                    if j < nb:
                        assert rel_err(g["p_d"][b, j], o["p_d"][b, j]) < PROB_RTOL, (b, j, g["p_d"][b, j], o["p_d"][b, j])
                        assert rel_err(g["q_d"][b, j], o["q_d"][b, j]) < PROB_RTOL, (b, j)
                else:
                    assert g["row_m"][b, j] == o["row_m"][b, j]
                    assert g["row_arg"][b, j] == o["row_arg"][b, j]
    if budget:
        assert excused <= int(1e-4 * max(decisions, 1)), f"{excused} excused of {decisions}"
    return decisions, excused


def gpu_to_numpy(res):
    return {k: v.detach().cpu().numpy() for k, v in res.items()}


# ---- per-request sampling parameters (top-k / top-p cuts) -------------------

def _probs(row, T):
    x = row.astype(np.float64)
    p = np.exp(x / T - (x / T).max())
    return p / p.sum()


def cut_ok(row, T, k, top_p, tau_gpu, tau_oracle):
    """(ok, excused): the GPU cut equals the oracle's, or lies within BAND of
    the top-p boundary (its mass above and at the cut straddle top_p)."""
    if tau_gpu == tau_oracle or (np.isnan(tau_gpu) and np.isnan(tau_oracle)):
        return True, False
    # a cut is the kept set {v : l_v >= tau}: two values that keep the same
    # tokens are the same cut (with nothing cut the GPU reports -inf, the
    # oracle the row's smallest logit)
    x32 = np.asarray(row, np.float32)
    if not np.isnan(tau_gpu) and not np.isnan(tau_oracle) and np.array_equal(x32 >= tau_gpu, x32 >= tau_oracle):
        return True, False
    if top_p >= 1.0:
        return False, False
    _, tau_k = oracle.truncate_row(row, T, k, 1.0)
    x = row.astype(np.float64)
    p = _probs(row, T)
    kept_k = x >= tau_k
    zk = p[kept_k].sum()
    above = p[kept_k & (x > tau_gpu)].sum() / zk
    incl = p[kept_k & (x >= tau_gpu)].sum() / zk
    ok = tau_gpu >= tau_k and np.any(x == tau_gpu) and above < top_p + BAND and incl >= top_p - BAND
    return bool(ok), True


def compare_sampling(g, o, rows, draft, T, k, p, tau_g, budget=True):
    """Verification under per-request (T, top_k, top_p): statuses equal; each
    decision identical, or excused when a row's top-p cut lies on the other
    side of its boundary (within BAND in mass) or the coin lies within BAND
    of the oracle's threshold / CDF interval.  Returns (decisions, excused)."""
    B, K1 = rows.shape[:2]
    decisions = excused = 0
    for b in range(B):
        assert g["status"][b] == o["status"][b], b
        if o["status"][b] != 0:
            continue
        Lg, Lo = int(g["accept_len"][b]), int(o["accept_len"][b])
        # the emitted token is always inside the cut of its row
        assert rows[b, Lg, g["out_token"][b]] >= tau_g[b, Lg], b
        decisions += min(Lg, Lo) + 2
        if Lg == Lo and g["out_token"][b] == o["out_token"][b]:
            continue
        other_side = False
        for j in range(min(Lg, Lo) + 1):
            ok, ex = cut_ok(rows[b, j], float(T[b]), int(k[b]), float(p[b]), float(tau_g[b, j]),
                            float(o["tau"][b, j]))
            assert ok, (b, j)
            other_side |= ex
        if other_side:  # a top-p cut on the other side of its boundary
            excused += 1
            continue
        if Lg != Lo:
            j = min(Lg, Lo)
            assert abs(o["u_acc"][b, j] - o["p_d"][b, j]) < BAND, (b, j, o["u_acc"][b, j], o["p_d"][b, j])
        else:
            pp, _ = oracle.truncate_row(rows[b, Lo], float(T[b]), int(k[b]), float(p[b]))
            r = pp.copy()
            if Lo < draft.shape[1]:
                r[draft[b, Lo]] = max(0.0, r[draft[b, Lo]] - 1.0)
            mass = r.sum()
            tok = int(g["out_token"][b])
            lo = r[:tok].sum() / mass
            hi = lo + r[tok] / mass
            assert r[tok] > 0 and lo - BAND <= o["u_res"][b] < hi + BAND, (b, tok, lo, hi, o["u_res"][b])
        excused += 1
    if budget:
        assert excused <= int(1e-4 * max(decisions, 1)), f"{excused} excused of {decisions}"
    return decisions, excused


# ---- draft trees -------------------------------------------------------------

def tree_children(fc, ns, n):
    out, c = [], fc[n]
    while c != -1:
        out.append(int(c))
        c = ns[c]
    return out


def compare_trees(g, o, rows, tok, fc, ns, T, seed, step, budget=True, seq_index=None):
    """Tree verification: statuses equal; accepted paths and emitted tokens
    identical, or excused when the depth's coin lies within BAND of a child's
    running-sum threshold or the final coin within BAND of the oracle's
    interval of the GPU's token.  Returns (decisions, excused)."""
    B = len(o["status"])
    decisions = excused = 0
    for b in range(B):
        assert g["status"][b] == o["status"][b], b
        if o["status"][b] != 0:
            continue
        Lg, Lo = int(g["accept_len"][b]), int(o["accept_len"][b])
        pg, po = list(g["path"][b, :Lg]), list(o["path"][b, :Lo])
        decisions += min(Lg, Lo) + 2
        if pg == po and g["out_token"][b] == o["out_token"][b]:
            # the emitted tokens: the path's tokens, then the out token
            assert list(g["emit"][b, :Lg + 1]) == [int(tok[b, n]) for n in pg] + [int(o["out_token"][b])]
            continue
        assert T > 0, f"greedy tree differs at b={b}"
        d = 0
        while d < min(Lg, Lo) and pg[d] == po[d]:
            d += 1
        node = 0 if d == 0 else po[d - 1]
        kids = tree_children(fc[b], ns[b], node)
        acc, lo, hi, _ = oracle.tree_node_info(rows[b, node], T, [int(tok[b, c]) for c in kids],
                                               int(g["out_token"][b]))
        ua, ur = oracle.uniforms(seed, step, b if seq_index is None else int(seq_index[b]), d)
        if d < Lg or d < Lo:  # the depth's coin against a running sum
            assert any(abs(ua - a) < BAND for a in acc), (b, d, ua, acc)
        else:  # same path, different final token
            assert lo - BAND <= ur < hi + BAND, (b, ur, lo, hi)
        excused += 1
    if budget:
        assert excused <= int(1e-4 * max(decisions, 1)), f"{excused} excused of {decisions}"
    return decisions, excused
