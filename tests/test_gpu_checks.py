"""The debug library (libsamspec_checks.so, built with SAMSPEC_CHECKS=1), in
which every index into a sequence's automaton arrays -- states, links,
out-token pool, transition hash, text, suffix chain -- is checked against
the array's extent before it is used.

On healthy inputs it must agree with the oracle bit for bit and raise no
check (the tiny workload token by token, every short string over two and
three letters, Zipf histories with their continuations, a long run of one
token).  A link planted outside its array in one sequence's automaton must
turn into status ST_BOUNDS for that sequence alone.  The planted index lands
in the next sequence's region of the workspace, so that even an unchecked
access would stay inside the caller's buffer."""
import itertools

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def checked(cuda_device):
    """The package with the debug library behind every SamBatch made here."""
    import sam_drafting_verification_gb300 as ss
    from sam_drafting_verification_gb300 import _binding
    lib = _binding.load(_binding.CHECKS_LIB_PATH)
    saved = _binding._lib
    _binding._lib = lib
    try:
        yield ss, _binding
    finally:
        _binding._lib = saved


def _i32(a, dev):
    return torch.as_tensor(np.ascontiguousarray(a, dtype=np.int32), device=dev)


def _same_states(batch, sam, b):
    g = batch.dump(b)
    o = sam.dump()
    assert g["status"] == 0, (b, g["status"])
    np.testing.assert_array_equal(g["len"], o["len"])
    np.testing.assert_array_equal(g["link"], o["link"])
    np.testing.assert_array_equal(g["min_endpos"], o["min_endpos"])
    np.testing.assert_array_equal(g["edges"], o["edges"])


def _same_drafts(out, sams, K):
    d, dl, ml, me = (t.cpu().numpy() for t in out)
    for b, sam in enumerate(sams):
        od, odl, oml, ome = sam.draft(K)
        assert (dl[b], ml[b], me[b]) == (odl, oml, ome), b
        np.testing.assert_array_equal(d[b], od)


def test_checked_build_on_short_strings(checked, cuda_device):
    ss, bd = checked
    strings = [s for n in range(1, 11) for s in itertools.product(range(2), repeat=n)]
    strings += [s for n in range(1, 7) for s in itertools.product(range(3), repeat=n)]
    B, C, K = len(strings), 10, 4
    toks = np.zeros((B, C), np.int32)
    lens = np.array([len(s) for s in strings], np.int32)
    for b, s in enumerate(strings):
        toks[b, :len(s)] = s
    batch = ss.SamBatch(B, C, 3, device=cuda_device)
    assert batch.lib is not None and batch.lib._name == bd.CHECKS_LIB_PATH
    batch.extend(_i32(toks, cuda_device), _i32(lens, cuda_device))
    out = batch.draft(K)
    assert (batch.status() == 0).all()
    sams = []
    for s in strings:
        sams.append(oracle.Sam(3))
        sams[-1].extend(np.array(s, np.int32))
    _same_drafts(out, sams, K)
    for b in range(0, B, 7):
        _same_states(batch, sams[b], b)


def test_checked_build_on_histories(checked, cuda_device):
    ss, bd = checked
    w = workloads.tiny()
    V, K = w["V"], w["K"]
    rng = np.random.default_rng(91)
    z = workloads.ZipfTokens(151936, 1.1)
    B, n, steps = 16, 4096, 40
    streams = [workloads.make_stream(rng, n + 4 * steps, 151936, 0.3, 8, 64, z) for _ in range(B - 1)]
    # one text with a run of 300 equal tokens: a suffix chain longer than the
    # kept chain, walked by link chasing
    run = np.concatenate([rng.integers(0, 50, 100), np.full(300, 7), rng.integers(0, 50, n + 4 * steps - 400)])
    streams.append(run.astype(np.int32))
    batch = ss.SamBatch(B, n + 4 * steps, 151936, device=cuda_device)
    hist = np.stack([s[:n] for s in streams])
    batch.extend(_i32(hist, cuda_device), _i32(np.full(B, n), cuda_device))
    sams = [oracle.Sam(151936) for _ in range(B)]
    for b in range(B):
        sams[b].extend(hist[b])
    pos = np.full(B, n)
    for s in range(steps):
        nn = rng.integers(1, 5, B).astype(np.int32)
        tk = np.stack([streams[b][pos[b]:pos[b] + 4] for b in range(B)]).astype(np.int32)
        out = batch.step(_i32(tk, cuda_device), _i32(nn, cuda_device), K)
        for b in range(B):
            sams[b].extend(tk[b, :nn[b]])
        _same_drafts(out, sams, K)
        pos += nn
    assert (batch.status() == 0).all()
    for b in (0, 5, B - 1):
        _same_states(batch, sams[b], b)
    # the tiny workload, token by token
    tb = ss.SamBatch(w["B"], 300, V, device=cuda_device)
    ts = [oracle.Sam(V) for _ in range(w["B"])]
    for t in range(w["hist"].shape[1]):
        tb.extend(_i32(w["hist"][:, t:t + 1], cuda_device), _i32(np.ones(w["B"]), cuda_device))
        for b in range(w["B"]):
            ts[b].extend(w["hist"][b, t:t + 1])
        _same_drafts(tb.draft(K), ts, K)
    assert (tb.status() == 0).all()


def _layout(B, C):
    """Offsets of the automata workspace regions (the library's layout)."""
    S, E = 2 * C + 1, 3 * C + 4
    H = 64
    while H < E + E // 2:
        H <<= 1
    P = 4 * E
    a = lambda x: (x + 255) & ~255  # noqa: E731
    off = {"states": 0}
    o = a(B * S * 16)
    off["links"] = o
    o = a(o + B * S * 4)
    off["chain"] = o
    o = a(o + B * 128 * 4)
    off["pool"] = o
    o = a(o + B * P * 4)
    off["hash"] = o
    o = a(o + B * H * 8)
    off["hist"] = o
    o = a(o + B * C * 4)
    off["scal"] = o
    off["total"] = a(o + B * 16 * 4)
    return S, off


def test_planted_link_outside_its_array(checked, cuda_device):
    ss, bd = checked
    B, C, V = 4, 64, 20
    rng = np.random.default_rng(5)
    toks = rng.integers(0, V, (B, 40)).astype(np.int32)
    batch = ss.SamBatch(B, C, V, device=cuda_device)
    batch.extend(_i32(toks, cuda_device), _i32(np.full(B, 40), cuda_device))
    assert (batch.status() == 0).all()
    S, off = _layout(B, C)
    assert off["total"] == batch.ws_bytes
    last1 = batch.dump(1)["last"]
    blob = batch.export()
    words = blob.view(torch.int32)
    # sequence 1: the link of its last state points S + 3 states on (into
    # sequence 2's links), and its suffix chain is marked as not kept, so the
    # next token's link walk follows that link
    words[(off["links"] // 4) + 1 * S + last1] = S + 3
    words[(off["scal"] // 4) + 1 * 16 + 8] = 0
    batch.import_(blob)
    more = rng.integers(0, V, (B, 2)).astype(np.int32)
    batch.step(_i32(more, cuda_device), _i32(np.full(B, 2), cuda_device), 3)
    st = batch.status()
    assert st[1] == bd.ST_BOUNDS, st
    assert st[0] == 0 and st[2] == 0 and st[3] == 0, st
    # the other sequences are intact: equal to the oracle's automata
    for b in (0, 2, 3):
        sam = oracle.Sam(V)
        sam.extend(np.concatenate([toks[b], more[b]]))
        _same_states(batch, sam, b)
