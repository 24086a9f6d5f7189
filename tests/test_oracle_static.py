"""Pins of the oracle's static-automaton matching (the volcengine.com
SAM-Decoding article, "Drafting with Suffix Automaton" and "Update of Suffix
Automaton": a corpus automaton stays fixed and a generated text is followed
by a matching state), checked against brute force: after every generated
token the match length is the length of the longest suffix of the generated
text that occurs in the corpus, the recorded end is the smallest end position
of that suffix in the corpus, and the draft copies the corpus after it."""
import numpy as np
import pytest

import oracle


def _longest_suffix_in(corpus, gen):
    """(length, smallest end position) of the longest suffix of gen that occurs
    in corpus; (0, -1) if none."""
    c = list(corpus)
    for L in range(len(gen), 0, -1):
        suf = list(gen[len(gen) - L:])
        ends = [i + L - 1 for i in range(len(c) - L + 1) if c[i:i + L] == suf]
        if ends:
            return L, min(ends)
    return 0, -1


@pytest.mark.parametrize("V,ncorpus,ngen", [(2, 30, 25), (3, 40, 25), (4, 60, 30), (8, 80, 40)])
def test_matching_state_equals_brute_force(V, ncorpus, ngen):
    rng = np.random.default_rng(V * 100 + ncorpus)
    K = 4
    for trial in range(25):
        corpus = rng.integers(0, V, ncorpus).astype(np.int32)
        if trial % 3 == 0:  # generated text that copies from the corpus, then drifts
            a = int(rng.integers(0, ncorpus - 10))
            gen = np.concatenate([corpus[a:a + 10], rng.integers(0, V, ngen - 10)]).astype(np.int32)
        else:
            gen = rng.integers(0, V, ngen).astype(np.int32)
        sam = oracle.Sam(V)
        sam.extend(corpus)
        state = (0, 0)
        for i in range(ngen):
            state, draft, dl, me = sam.match(state, gen[i:i + 1], K)
            L, e = _longest_suffix_in(corpus, gen[:i + 1])
            assert state[1] == L, (trial, i)
            assert me == e, (trial, i)
            want = [] if L == 0 else list(corpus[e + 1:e + 1 + K])
            assert dl == len(want) and list(draft[:dl]) == want
            assert all(draft[dl:] == -1)


def test_incremental_equals_one_call():
    rng = np.random.default_rng(7)
    corpus = rng.integers(0, 5, 200).astype(np.int32)
    gen = np.concatenate([corpus[50:90], rng.integers(0, 5, 30)]).astype(np.int32)
    sam = oracle.Sam(5)
    sam.extend(corpus)
    st = (0, 0)
    for i in range(0, len(gen), 7):
        st, d1, l1, m1 = sam.match(st, gen[i:i + 7], 3)
    st2, d2, l2, m2 = sam.match((0, 0), gen, 3)
    assert st == st2 and l1 == l2 and m1 == m2 and list(d1) == list(d2)


def test_eos_joined_documents():
    # documents joined by an end-of-sequence token: a match may not reach
    # across a document boundary unless the generated text holds that token
    eos = 0
    docs = [[1, 2, 3, 4], [2, 3, 5, 6], [3, 4, 7]]
    corpus = np.array([t for d in docs for t in d + [eos]], np.int32)
    sam = oracle.Sam(8)
    sam.extend(corpus)
    (v, l), draft, dl, me = sam.match((0, 0), [2, 3], 3)
    assert l == 2 and me == 2 and list(draft[:dl]) == [4, 0, 2]
    (v, l), draft, dl, me = sam.match((0, 0), [9 % 8, 2, 3, 5], 2)  # 1 2 3 5: only "2 3 5" occurs
    assert l == 3 and list(draft[:dl]) == [6, 0]


def test_selection_prefers_the_dynamic_draft():
    assert oracle.select_static(10, 3, 2) is True
    assert oracle.select_static(5, 3, 2) is False   # longer by 2, not by more than 2
    assert oracle.select_static(3, 3, 1) is False
    assert oracle.select_static(0, 0, 1) is False
