"""Pins of the oracle's suffix automaton against facts the pages and the
mathematics fix (no GPU).

* the ABCBC worked example of "SAM投机推理：长序列强化学习训练加速利器" §1.1
  (endpos(BC) = {2,4}; the draft after the final C is "BC");
* brute force on every string over 2 letters up to length 12 and over 3 letters
  up to length 8: longest earlier-occurring suffix, its first end position, the
  draft that follows it, the number of endpos classes and of distinct
  substrings;
* structural invariants (suffix-link lengths, state and transition bounds,
  linear total link-walk work) on long synthetic streams.
"""
import itertools
import os

import numpy as np
import pytest

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "abcbc.txt")


def _read_golden():
    kv = {}
    for line in open(GOLDEN, encoding="utf-8"):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        k, v = line.split("=", 1)
        kv[k.strip()] = v.strip()
    return kv


def _endpos_of_state(dump, v):
    """endpos(v) from the automaton: the end positions i whose prefix state
    (the state created when s_i was appended, len = i + 1 and min_endpos = i)
    lies in v's subtree of the suffix-link tree."""
    ln, lk, me = dump["len"], dump["link"], dump["min_endpos"]
    out = set()
    for u in range(1, len(ln)):
        if me[u] != ln[u] - 1:
            continue  # a clone: its min_endpos comes from the state it split
        w = u
        while w != -1 and w != v:
            w = lk[w]
        if w == v:
            out.add(int(me[u]))
    return out


def _walk(dump, tokens):
    nxt = {(int(s), int(t)): int(to) for s, t, to in dump["edges"]}
    v = 0
    for t in tokens:
        v = nxt[(v, t)]
    return v


def test_abcbc_worked_example():
    g = _read_golden()
    letters = {"A": 0, "B": 1, "C": 2}
    s = [letters[c] for c in g["string"]]
    sam = oracle.Sam(3)
    assert sam.extend(s) == 0
    dump = sam.dump()
    v_bc = _walk(dump, [letters["B"], letters["C"]])
    assert _endpos_of_state(dump, v_bc) == {int(x) for x in g["endpos_BC"].split()}
    # the printed example: from the last node the link walk stops at node BC
    draft, dl, ml, me = sam.draft(3)
    assert [int(x) for x in draft[:dl]] == [letters[c] for c in g["draft_after_final_C"]]
    assert ml == 2 and me == min(int(x) for x in g["endpos_BC"].split())
    last = sam.sizes()["last"]
    assert dump["link"][last] == v_bc  # the walk reaches node BC in one link step


def _brute(s, K):
    """Longest suffix w of s (|w| < n) that also ends at an earlier position,
    the smallest such earlier end e, and the draft s[e+1 : e+1+K]."""
    n = len(s)
    for ell in range(n - 1, 0, -1):
        w = s[n - ell:]
        for e in range(ell - 1, n - 1):
            if s[e - ell + 1:e + 1] == w:
                return ell, e, s[e + 1:e + 1 + K]
    return 0, -1, []


def _brute_classes(s):
    """(#distinct non-empty substrings, #distinct endpos sets among them)."""
    n = len(s)
    endpos = {}
    for i in range(n):
        for j in range(i, n):
            endpos.setdefault(tuple(s[i:j + 1]), set()).add(j)
    return len(endpos), len({frozenset(e) for e in endpos.values()})


def _check_string(s, V, K=4):
    sam = oracle.Sam(V)
    assert sam.extend(s) == 0
    draft, dl, ml, me = sam.draft(K)
    ell, e, want = _brute(list(s), K)
    assert (ml, me if ell else -1) == (ell, e), s
    assert list(draft[:dl]) == list(want), s
    assert all(x == -1 for x in draft[dl:])
    dump = sam.dump()
    ln, lk = dump["len"], dump["link"]
    n_sub, n_cls = _brute_classes(list(s))
    assert len(ln) - 1 == n_cls, s
    assert int(sum(ln[v] - ln[lk[v]] for v in range(1, len(ln)))) == n_sub, s


@pytest.mark.parametrize("V,maxlen", [(2, 12), (3, 8)])
def test_bruteforce_every_small_string(V, maxlen):
    for n in range(1, maxlen + 1):
        for s in itertools.product(range(V), repeat=n):
            _check_string(s, V)


def test_bruteforce_draft_after_every_token():
    rng = np.random.default_rng(7)
    for trial in range(40):
        V = int(rng.integers(2, 9))
        n = int(rng.integers(1, 60))
        s = workloads.make_stream(rng, n, V, 0.3, 2, 6)
        sam = oracle.Sam(V)
        for i in range(n):
            sam.extend([int(s[i])])
            K = int(rng.integers(1, 6))
            draft, dl, ml, me = sam.draft(K)
            ell, e, want = _brute(list(s[:i + 1]), K)
            assert ml == ell and (me == e if ell else me == -1)
            assert list(draft[:dl]) == list(want)


@pytest.mark.parametrize("seed,n,V,zipf", [(11, 20000, 64, False), (12, 20000, 50000, True)])
def test_invariants_long_stream(seed, n, V, zipf):
    rng = np.random.default_rng(seed)
    z = workloads.ZipfTokens(V) if zipf else None
    s = workloads.make_stream(rng, n, V, 0.4, 8, 64, z)
    sam = oracle.Sam(V)
    assert sam.extend(s) == 0
    sz = sam.sizes()
    d = sam.dump()
    ln, lk, me = d["len"], d["link"], d["min_endpos"]
    assert sz["n_states"] <= max(2, 2 * n - 1)
    assert sz["n_edges"] <= 3 * n - 4
    assert np.all(ln[lk[1:]] < ln[1:])
    assert lk[0] == -1 and np.all(lk[1:] >= 0)
    # every state's strings end first at min_endpos: the longest one read
    # there matches the text, and so does every transition target's
    for v in range(1, sz["n_states"]):
        assert ln[v] - 1 <= me[v] < n
    edges = d["edges"]
    # transition (v, c) -> w: w's strings end one position after some
    # occurrence of v's strings followed by c, so min_endpos(w) >= min_endpos(v) + 1
    assert np.all(me[edges[:, 2]] >= me[edges[:, 0]] + 1)
    # amortised O(1) per extension: total link-walk work linear in n
    assert sz["walk_steps"] <= 4 * n


def test_extend_rejects_out_of_range_token():
    sam = oracle.Sam(4)
    assert sam.extend([0, 1, 2]) == 0
    assert sam.extend([4]) == oracle.ETOKEN
    assert sam.extend([-1]) == oracle.ETOKEN
    assert sam.sizes()["n_tokens"] == 3


def test_empty_and_single_token():
    sam = oracle.Sam(4)
    draft, dl, ml, me = sam.draft(3)
    assert (dl, ml, me) == (0, 0, -1) and list(draft) == [-1, -1, -1]
    sam.extend([2])
    draft, dl, ml, me = sam.draft(3)
    assert (dl, ml, me) == (0, 0, -1)
    sam.extend([2])  # "cc": suffix "c" ends earlier at 0, followed by c
    draft, dl, ml, me = sam.draft(3)
    assert (dl, ml, me) == (1, 1, 0) and list(draft[:1]) == [2]
