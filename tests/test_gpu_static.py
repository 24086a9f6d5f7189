"""Static use of a device automaton (a corpus) against the oracle: matching
states (state id and length), drafts and first ends after every step; the
adaptive choice between dynamic and static drafts."""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ss(cuda_device):
    import sam_drafting_verification_gb300 as ss
    return ss


def _i32(a, dev):
    return torch.as_tensor(np.ascontiguousarray(a, dtype=np.int32), device=dev)


def _corpus_batch(ss, corpus, V, dev):
    cb = ss.SamBatch(1, len(corpus), V, device=dev)
    cb.extend(_i32(corpus[None, :], dev), _i32([len(corpus)], dev))
    assert cb.status()[0] == 0
    return cb


def _follow(ss, dev, corpus, V, gens, K, chunks):
    """Matches every generated text step by step on the device and with the
    oracle; returns the number of steps compared."""
    n = len(gens)
    cb = _corpus_batch(ss, corpus, V, dev)
    osam = oracle.Sam(V)
    osam.extend(corpus)
    state = torch.zeros((n, 2), dtype=torch.int32, device=dev)
    ostate = [(0, 0)] * n
    pos = np.zeros(n, np.int64)
    rng = np.random.default_rng(len(corpus))
    steps = 0
    while any(pos[i] < len(gens[i]) for i in range(n)):
        k = np.array([min(int(rng.integers(1, chunks + 1)), len(gens[i]) - pos[i]) for i in range(n)], np.int32)
        toks = np.zeros((n, chunks), np.int32)
        for i in range(n):
            toks[i, :k[i]] = gens[i][pos[i]:pos[i] + k[i]]
        d, dl, ml, me = (t.cpu().numpy() for t in cb.match(0, state, _i32(toks, dev), _i32(k, dev), K))
        st = state.cpu().numpy()
        for i in range(n):
            ostate[i], od, odl, ome = osam.match(ostate[i], toks[i, :k[i]], K)
            assert tuple(st[i]) == ostate[i], (steps, i, tuple(st[i]), ostate[i])
            assert ml[i] == ostate[i][1] and me[i] == ome and dl[i] == odl, (steps, i)
            np.testing.assert_array_equal(d[i], od)
        pos += k
        steps += 1
    return steps


@pytest.mark.parametrize("V,n", [(2, 40), (4, 120), (8, 300)])
def test_small_alphabets(ss, cuda_device, V, n):
    rng = np.random.default_rng(V)
    corpus = rng.integers(0, V, n).astype(np.int32)
    gens = []
    for i in range(12):
        a = int(rng.integers(0, n - 20))
        gens.append(np.concatenate([corpus[a:a + 15], rng.integers(0, V, 25)]).astype(np.int32))
    assert _follow(ss, cuda_device, corpus, V, gens, 5, 3) > 0


def test_zipf_corpus_of_documents(ss, cuda_device):
    """A 20k-token corpus of documents joined by an end-of-sequence token
    (Zipf(1.1) tokens, copied spans), 48 generated texts that copy corpus
    passages and drift, followed 1-4 tokens per step, K = 6."""
    V = 151936
    eos = V - 1  # a token the Zipf draws almost never produce
    rng = np.random.default_rng(55)
    z = workloads.ZipfTokens(V, 1.1)
    docs = [workloads.make_stream(rng, int(rng.integers(200, 900)), V, 0.3, 8, 64, z) for _ in range(40)]
    corpus = np.concatenate([np.concatenate([d, [eos]]) for d in docs]).astype(np.int32)
    gens = []
    for i in range(48):
        parts = []
        for _ in range(4):
            a = int(rng.integers(0, len(corpus) - 80))
            parts.append(corpus[a:a + int(rng.integers(10, 60))])
            parts.append(z.draw(rng, int(rng.integers(1, 6))).astype(np.int32))
        gens.append(np.concatenate(parts).astype(np.int32))
    assert _follow(ss, cuda_device, corpus, V, gens, 6, 4) > 0


def test_out_of_range_state_and_token(ss, cuda_device):
    V = 10
    corpus = np.array([1, 2, 3, 1, 2, 4], np.int32)
    cb = _corpus_batch(ss, corpus, V, cuda_device)
    state = _i32([[-5, 3], [2, 2], [999, 1]], cuda_device)
    toks = _i32([[1, 2], [V, 0], [1, 2]], cuda_device)
    d, dl, ml, me = cb.match(0, state, toks, _i32([2, 1, 2], cuda_device), 3)
    st = state.cpu().numpy()
    osam = oracle.Sam(V)
    osam.extend(corpus)
    want, _, _, _ = osam.match((0, 0), [1, 2], 3)
    assert tuple(st[0]) == want and tuple(st[2]) == want  # restarted from the root
    assert tuple(st[1]) == (0, 0) and dl.cpu().numpy()[1] == 0  # token V matches nothing


def test_select_drafts_matches_oracle_rule(ss, cuda_device):
    rng = np.random.default_rng(4)
    n, K, bias = 500, 4, 2
    dyn = (rng.integers(0, 100, (n, K)), rng.integers(0, K + 1, n), rng.integers(0, 12, n))
    st = (rng.integers(0, 100, (n, K)), rng.integers(0, K + 1, n), rng.integers(0, 12, n))
    d, dl, src = ss.select_drafts(tuple(_i32(x, cuda_device) for x in dyn),
                                  tuple(_i32(x, cuda_device) for x in st), bias)
    d, dl, src = d.cpu().numpy(), dl.cpu().numpy(), src.cpu().numpy()
    for i in range(n):
        use = oracle.select_static(int(st[2][i]), int(dyn[2][i]), bias)
        assert src[i] == int(use)
        pick = st if use else dyn
        assert dl[i] == pick[1][i] and list(d[i]) == list(pick[0][i])
