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
