"""GPU parity of the device suffix automata against the oracle, through the
C ABI: state arrays (len, link, min_endpos) and sorted transition triples
bit-exact, drafts / match lengths / min_endpos bit-exact after every step."""
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


def _check_states(batch, sams, which):
    for b in which:
        g = batch.dump(b)
        o = sams[b].dump()
        assert g["status"] == 0, (b, g["status"])
        assert g["n_states"] == len(o["len"]) and g["n_edges"] == len(o["edges"]), b
        np.testing.assert_array_equal(g["len"], o["len"])
        np.testing.assert_array_equal(g["link"], o["link"])
        np.testing.assert_array_equal(g["min_endpos"], o["min_endpos"])
        np.testing.assert_array_equal(g["edges"], o["edges"])


def _check_drafts(out, sams, K, which):
    d, dl, ml, me = (t.cpu().numpy() for t in out)
    for b in which:
        od, odl, oml, ome = sams[b].draft(K)
        assert (dl[b], ml[b], me[b]) == (odl, oml, ome), (b, (dl[b], ml[b], me[b]), (odl, oml, ome))
        np.testing.assert_array_equal(d[b], od)


def test_abcbc_on_device(ss, cuda_device):
    batch = ss.SamBatch(1, 16, 3, device=cuda_device)
    batch.extend(_i32([[0, 1, 2, 1, 2]], cuda_device), _i32([5], cuda_device))
    d, dl, ml, me = batch.draft(3)
    assert d.cpu().tolist() == [[1, 2, -1]] and dl.item() == 2 and ml.item() == 2 and me.item() == 2
    g = batch.dump(0)
    assert g["len"].tolist() == [0, 1, 2, 3, 4, 1, 5, 2]
    assert g["link"].tolist() == [-1, 0, 5, 7, 5, 0, 7, 0]
    assert g["min_endpos"].tolist() == [-1, 0, 1, 2, 3, 1, 4, 2]


def test_tiny_token_by_token(ss, cuda_device):
    w = workloads.tiny()
    B, V, K = w["B"], w["V"], w["K"]
    hist = w["hist"]
    batch = ss.SamBatch(B, hist.shape[1] + 8, V, device=cuda_device)
    sams = [oracle.Sam(V) for _ in range(B)]
    rng = np.random.default_rng(5)
    pos = np.zeros(B, np.int64)
    while (pos < hist.shape[1]).any():
        n_new = np.minimum(rng.integers(0, 5, size=B), hist.shape[1] - pos).astype(np.int32)
        toks = np.full((B, 4), -7, np.int32)
        for b in range(B):
            toks[b, :n_new[b]] = hist[b, pos[b]:pos[b] + n_new[b]]
            sams[b].extend(toks[b, :n_new[b]])
        out = batch.step(_i32(toks, cuda_device), _i32(n_new, cuda_device), K)
        _check_drafts(out, sams, K, range(B))
        pos += n_new
    _check_states(batch, sams, range(B))


@pytest.mark.parametrize("V,p_copy,n", [(2, 0.2, 3000), (5, 0.5, 3000), (64, 0.3, 5000)])
def test_small_alphabets_bulk(ss, cuda_device, V, p_copy, n):
    rng = np.random.default_rng(V)
    B = 6
    hist = np.stack([workloads.make_stream(rng, n, V, p_copy, 2, 40) for _ in range(B)])
    batch = ss.SamBatch(B, n, V, device=cuda_device)
    batch.extend(_i32(hist, cuda_device), _i32(np.full(B, n), cuda_device))
    sams = [oracle.Sam(V) for _ in range(B)]
    for b in range(B):
        sams[b].extend(hist[b])
    _check_states(batch, sams, range(B))
    _check_drafts(batch.draft(7), sams, 7, range(B))


def test_rs_bf16_b64_histories(ss, cuda_device):
    """B=64, V=151936, 4096-token Zipf histories: bulk build then 40 steps of
    1-4 tokens; drafts of every sequence after every step, full state arrays of
    a sample of sequences at the end."""
    w = workloads.rs_bf16_b64(with_logits=False)
    B, V, K = w["B"], w["V"], w["K"]
    hist = w["hist"]
    rng = np.random.default_rng(9)
    steps = 40
    extra = workloads.make_stream(rng, steps * 4 * B, V, 0.3, 8, 64, workloads.ZipfTokens(V)).reshape(B, -1)
    batch = ss.SamBatch(B, hist.shape[1] + extra.shape[1], V, device=cuda_device)
    batch.extend(_i32(hist, cuda_device), _i32(np.full(B, hist.shape[1]), cuda_device))
    sams = [oracle.Sam(V) for _ in range(B)]
    for b in range(B):
        sams[b].extend(hist[b])
    _check_drafts(batch.draft(K), sams, K, range(B))
    pos = np.zeros(B, np.int64)
    for s in range(steps):
        n_new = rng.integers(1, 5, size=B).astype(np.int32)
        toks = np.stack([extra[b, pos[b]:pos[b] + 4] for b in range(B)]).astype(np.int32)
        for b in range(B):
            sams[b].extend(toks[b, :n_new[b]])
        out = batch.step(_i32(toks, cuda_device), _i32(n_new, cuda_device), K)
        _check_drafts(out, sams, K, range(B))
        pos += n_new
    _check_states(batch, sams, [0, 17, 33, 63])


def test_long_rollout_all_sequences(ss, cuda_device):
    """B=256 histories log-uniform in [16k, 32k] (copy prob 0.5, spans 16-256):
    prefill, then 512 steps of U{1..4} tokens + K=3 drafts.  The oracle
    follows all 256 sequences: drafts, draft lengths, match lengths and first
    ends after every step, and the full state arrays and transition triples
    of 32 of them at the end; every sequence must stay healthy."""
    w = workloads.long_rollout()
    B, V, K, steps = w["B"], w["V"], w["K"], w["steps"]
    lens, n_new, streams = w["lens"], w["n_new"], w["streams"]
    cap = int(max(len(s) for s in streams))
    batch = ss.SamBatch(B, cap, V, device=cuda_device)
    maxlen = int(lens.max())
    pre = np.zeros((B, maxlen), np.int32)
    for b in range(B):
        pre[b, :lens[b]] = streams[b][:lens[b]]
    batch.extend(_i32(pre, cuda_device), _i32(lens, cuda_device))
    sams = [oracle.Sam(V) for _ in range(B)]
    for b in range(B):
        sams[b].extend(streams[b][:lens[b]])
    pos = lens.astype(np.int64).copy()
    toks = np.zeros((steps, B, 4), np.int32)
    for s in range(steps):
        for b in range(B):
            k = n_new[s, b]
            toks[s, b, :k] = streams[b][pos[b]:pos[b] + k]
        pos += n_new[s]
    toks_d = _i32(toks, cuda_device)
    nn_d = _i32(n_new, cuda_device)
    for s in range(steps):
        d, dl, ml, me = (t.cpu().numpy() for t in batch.step(toks_d[s], nn_d[s], K))
        od, info = oracle.step_batch(sams, toks[s], n_new[s], K)
        np.testing.assert_array_equal(dl, info[:, 0], err_msg=f"draft_len, step {s}")
        np.testing.assert_array_equal(ml, info[:, 1], err_msg=f"match_len, step {s}")
        np.testing.assert_array_equal(me, info[:, 2], err_msg=f"min_endpos, step {s}")
        np.testing.assert_array_equal(d, od, err_msg=f"drafts, step {s}")
    assert (batch.status() == 0).all()
    _check_states(batch, sams, list(range(0, B, 8)))


def test_errors_freeze_one_sequence(ss, cuda_device):
    V = 16
    batch = ss.SamBatch(4, 10, V, device=cuda_device)
    toks = np.array([[1, 2, 3, 1, 2, 3, 1, 2, 3, 1, 2, 3],   # exceeds capacity 10
                     [1, 2, 16, 1, 0, 0, 0, 0, 0, 0, 0, 0],  # token 16 >= V
                     [1, 2, 1, 2, 1, 2, 1, 0, 0, 0, 0, 0],   # fine
                     [3, 3, 3, 0, 0, 0, 0, 0, 0, 0, 0, 0]], np.int32)
    n_new = np.array([12, 4, 7, 13], np.int32)  # 13 > max_new for sequence 3
    batch.extend(_i32(toks, cuda_device), _i32(n_new, cuda_device))
    st = batch.status()
    assert st.tolist() == [ss.ST_CAPACITY, ss.ST_TOKEN, 0, ss.ST_BADDRAFT]
    d, dl, ml, me = batch.draft(3)
    dl = dl.cpu().numpy()
    assert dl[0] == 0 and dl[1] == 0 and dl[3] == 0
    o = oracle.Sam(V)
    o.extend(toks[2, :7])
    od, odl, oml, ome = o.draft(3)
    assert dl[2] == odl and d[2].cpu().tolist() == od.tolist()
    # frozen sequences ignore further tokens; reset revives them
    batch.reset(_i32([1, 1, 0, 1], cuda_device))
    assert batch.status().tolist() == [0, 0, 0, 0]
    batch.extend(_i32(toks[:, :3], cuda_device), _i32([3, 2, 0, 3], cuda_device))
    g = batch.dump(0)
    assert g["n_tokens"] == 3 and g["status"] == 0


def test_empty_sequences_and_export_import(ss, cuda_device):
    V = 8
    batch = ss.SamBatch(3, 64, V, device=cuda_device)
    d, dl, ml, me = batch.draft(4)
    assert dl.cpu().tolist() == [0, 0, 0] and me.cpu().tolist() == [-1, -1, -1]
    assert (d.cpu() == -1).all()
    rng = np.random.default_rng(3)
    toks = rng.integers(0, V, size=(3, 40)).astype(np.int32)
    batch.extend(_i32(toks, cuda_device), _i32([40, 20, 0], cuda_device))
    snap = batch.export()
    before = [batch.dump(b) for b in range(3)]
    batch.extend(_i32(toks, cuda_device), _i32([10, 10, 10], cuda_device))
    batch.import_(snap)
    after = [batch.dump(b) for b in range(3)]
    for x, y in zip(before, after):
        for k in ("len", "link", "min_endpos", "edges"):
            np.testing.assert_array_equal(x[k], y[k])


def test_host_argument_errors(ss, cuda_device):
    with pytest.raises(ss.SamspecError):
        ss.SamBatch(0, 10, 10, device=cuda_device)
    with pytest.raises(ss.SamspecError):
        ss.SamBatch(1, 10, 1 << 19, device=cuda_device)
    batch = ss.SamBatch(2, 10, 10, device=cuda_device)
    with pytest.raises(ss.SamspecError):
        batch.draft(65)


def test_long_suffix_chains(ss, cuda_device):
    """Texts whose suffix chains grow past 128 states (long runs of one token,
    short periods) and shrink again, built in bulk and in steps of 1-4
    tokens: states, transitions and drafts stay bit-exact."""
    rng = np.random.default_rng(77)
    V = 50
    texts = [
        np.concatenate([np.full(400, 7), rng.integers(0, V, 300)]),
        np.concatenate([np.tile([3, 4], 250), rng.integers(0, V, 200), np.tile([3, 4], 100)]),
        np.concatenate([np.tile([1, 2, 3], 120), np.full(150, 9), np.tile([1, 2, 3], 60)]),
        workloads.make_stream(rng, 900, V, 0.6, 64, 200),
    ]
    n = max(len(t) for t in texts)
    B = len(texts)
    hist = np.zeros((B, n), np.int32)
    for b, t in enumerate(texts):
        hist[b, :len(t)] = t
    lens = np.array([len(t) for t in texts], np.int32)
    sams = [oracle.Sam(V) for _ in range(B)]
    for b in range(B):
        sams[b].extend(texts[b])
    bulk = ss.SamBatch(B, n, V, device=cuda_device)
    bulk.extend(_i32(hist, cuda_device), _i32(lens, cuda_device))
    _check_states(bulk, sams, range(B))
    _check_drafts(bulk.draft(5), sams, 5, range(B))
    step = ss.SamBatch(B, n, V, device=cuda_device)
    ref = [oracle.Sam(V) for _ in range(B)]
    pos = np.zeros(B, np.int64)
    while (pos < lens).any():
        k = np.minimum(rng.integers(1, 5, size=B), lens - pos).astype(np.int32)
        toks = np.zeros((B, 4), np.int32)
        for b in range(B):
            toks[b, :k[b]] = texts[b][pos[b]:pos[b] + k[b]]
            ref[b].extend(toks[b, :k[b]])
        out = step.step(_i32(toks, cuda_device), _i32(k, cuda_device), 5)
        _check_drafts(out, ref, 5, range(B))
        pos += k
    _check_states(step, ref, range(B))
