"""GPU parity of spec_verify against the oracle through the C ABI: greedy
decisions bit-exact; rejection-sampling decisions identical up to the excused
rounding band; probabilities within 1e-6 relative.  Covers the tiny case, the
B=64 bf16 T=1 SAM-draft workload, the draft-model workload, the B=1024 sweep
(sampled sequences at full size), ragged and unaligned vocabularies, and
malformed inputs."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import compare_verify, gpu_to_numpy

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ss(cuda_device):
    import sam_drafting_verification_gb300 as ss
    return ss


def _run_both(ss, dev, target_f32, draft, draft_len=None, T=0.0, seed=0, step=0, draft_logits=None,
              t_dtype=torch.float32, d_dtype=torch.float32):
    """Runs GPU and oracle on the same values (bf16 inputs rounded first)."""
    tt = torch.from_numpy(np.ascontiguousarray(target_f32)).to(t_dtype)
    tg = tt.to(dev)
    t_exact = tt.float().numpy()
    dg = None
    d_exact = None
    if draft_logits is not None:
        dd = torch.from_numpy(np.ascontiguousarray(draft_logits)).to(d_dtype)
        dg = dd.to(dev)
        d_exact = dd.float().numpy()
    dr = torch.as_tensor(np.ascontiguousarray(draft, np.int32), device=dev)
    dl = None if draft_len is None else torch.as_tensor(np.asarray(draft_len, np.int32), device=dev)
    g = gpu_to_numpy(ss.spec_verify(tg, dr, dl, temperature=T, seed=seed, step=step,
                                    draft_logits=dg, emit=True, debug=True))
    o = oracle.verify(t_exact, draft, draft_len, temperature=T, seed=seed, step=step,
                      draft_logits=d_exact if T > 0 else None)
    return g, o, t_exact, d_exact


def _check(g, o, t_exact, d_exact, draft, draft_len, T):
    dec, exc = compare_verify(g, o, lambda b: t_exact[b], draft, draft_len, T,
                              None if d_exact is None else (lambda b: d_exact[b]))
    # emit = accepted drafts then the out token
    B, K = draft.shape
    for b in range(B):
        L = g["accept_len"][b]
        if L < 0:
            assert g["emit_len"][b] == 0
            continue
        assert g["emit_len"][b] == L + 1
        assert list(g["emit"][b, :L]) == list(draft[b, :L])
        assert g["emit"][b, L] == g["out_token"][b]
    return dec, exc


def test_uniforms_match_oracle(ss, cuda_device):
    B, K = 37, 5
    for seed, step in [(0, 0), (12345, 7), (2**64 - 1, 2**40 + 3)]:
        u = ss.spec_uniforms(B, K, seed, step, cuda_device).cpu().numpy().astype(np.float64)
        for b in range(B):
            for j in range(K + 1):
                assert tuple(u[b, j]) == oracle.uniforms(seed, step, b, j)


def test_tiny_greedy(ss, cuda_device):
    w = workloads.tiny()
    sams = [oracle.Sam(w["V"]) for _ in range(w["B"])]
    draft = np.zeros((w["B"], w["K"]), np.int32)
    dlen = np.zeros(w["B"], np.int32)
    for b in range(w["B"]):
        sams[b].extend(w["hist"][b])
        d, dl, _, _ = sams[b].draft(w["K"])
        draft[b] = np.maximum(d, 0)
        dlen[b] = dl
    g, o, te, de = _run_both(ss, cuda_device, w["logits"], draft, dlen, T=0.0)
    _check(g, o, te, de, draft, dlen, 0.0)
    assert (g["accept_len"] == o["accept_len"]).all() and (g["out_token"] == o["out_token"]).all()


@pytest.mark.parametrize("K", [1, 3, 5, 8])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_greedy_random(ss, cuda_device, K, dtype):
    rng = np.random.default_rng(100 + K)
    B, V = 48, 20000
    logits, draft = workloads.sweep_host(100 + K, B, K, V)
    # half of the sequences draft the argmax so that long chains occur
    am = np.argmax(logits[:, :K], axis=-1).astype(np.int32)
    draft[::2] = am[::2]
    dlen = rng.integers(0, K + 1, size=B).astype(np.int32)
    g, o, te, de = _run_both(ss, cuda_device, logits, draft, dlen, T=0.0, t_dtype=dtype)
    _check(g, o, te, de, draft, dlen, 0.0)


@pytest.mark.parametrize("T", [0.3, 1.0, 2.0])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_sampling_one_hot(ss, cuda_device, T, dtype):
    B, K, V = 64, 4, 40000
    logits, draft = workloads.sweep_host(200, B, K, V)
    am = np.argmax(logits[:, :K], axis=-1).astype(np.int32)
    draft[::3] = am[::3]
    g, o, te, de = _run_both(ss, cuda_device, logits, draft, None, T=T, seed=11, step=3, t_dtype=dtype)
    _check(g, o, te, de, draft, None, T)


def test_rs_bf16_b64_workload(ss, cuda_device):
    """B=64, V=151936, bf16 N(0, sd 2) + 4 on the truth, SAM drafts (K=3) from
    the oracle's automaton over each 4096-token history, T=1.0."""
    w = workloads.rs_bf16_b64()
    B, K = w["B"], w["K"]
    draft = np.zeros((B, K), np.int32)
    dlen = np.zeros(B, np.int32)
    for b in range(B):
        s = oracle.Sam(w["V"])
        s.extend(w["hist"][b])
        d, dl, _, _ = s.draft(K)
        draft[b] = np.maximum(d, 0)
        dlen[b] = dl
    for step in range(3):
        g, o, te, de = _run_both(ss, cuda_device, w["logits"], draft, dlen, T=1.0, seed=1002,
                                 step=step, t_dtype=torch.bfloat16)
        _check(g, o, te, de, draft, dlen, 1.0)


@pytest.mark.parametrize("tdt,ddt", [(torch.float32, torch.float32), (torch.bfloat16, torch.bfloat16),
                                     (torch.float32, torch.bfloat16), (torch.bfloat16, torch.float32)])
def test_draft_model_workload(ss, cuda_device, tdt, ddt):
    """B=32, K=5, V=151936, draft logits = target + N(0,1), drafts sampled from
    softmax(draft/0.7), T=0.7, residual max(0, p - q) resampling."""
    w = workloads.draft_model()
    g, o, te, de = _run_both(ss, cuda_device, w["target"], w["draft"], None, T=w["temperature"],
                             seed=1003, step=1, draft_logits=w["draft_logits"], t_dtype=tdt, d_dtype=ddt)
    _check(g, o, te, de, w["draft"], None, w["temperature"])
    assert (g["accept_len"] > 0).any()


@pytest.mark.parametrize("V", [8, 1000, 50000, 50257, 151936])
def test_ragged_and_unaligned_vocab(ss, cuda_device, V):
    B, K = 9, 3
    logits, draft = workloads.sweep_host(300 + V, B, K, V)
    for T in (0.0, 1.0):
        for dtype in (torch.float32, torch.bfloat16):
            g, o, te, de = _run_both(ss, cuda_device, logits, draft, None, T=T, seed=5, t_dtype=dtype)
            _check(g, o, te, de, draft, None, T)
    dlog = (logits[:, :K] + workloads.gaussian_logits(np.random.default_rng(V), (B, K, V), 1.0)).astype(np.float32)
    g, o, te, de = _run_both(ss, cuda_device, logits, draft, None, T=0.8, seed=6, draft_logits=dlog)
    _check(g, o, te, de, draft, None, 0.8)


def test_bonus_only_and_all_accepted(ss, cuda_device):
    B, K, V = 16, 4, 30000
    logits, _ = workloads.sweep_host(400, B, K, V)
    am = np.argmax(logits[:, :K], axis=-1).astype(np.int32)
    # draft_len 0: the bonus row only
    for T in (0.0, 1.0):
        g, o, te, de = _run_both(ss, cuda_device, logits, am, np.zeros(B, np.int32), T=T)
        _check(g, o, te, de, am, np.zeros(B, np.int32), T)
        assert (g["accept_len"] == 0).all()
    # greedy with argmax drafts: every draft accepted, bonus from the last row
    g, o, te, de = _run_both(ss, cuda_device, logits, am, None, T=0.0)
    assert (g["accept_len"] == K).all()
    assert (g["out_token"] == np.argmax(logits[:, K], axis=-1)).all()


def test_malformed_rows_and_drafts(ss, cuda_device):
    B, K, V = 8, 2, 5000
    logits, draft = workloads.sweep_host(500, B, K, V)
    am = np.argmax(logits[:, :K], axis=-1).astype(np.int32)
    draft[:] = am
    logits[0, 0, 17] = np.nan
    logits[1, 0, :] = -np.inf
    logits[2, 0, 3] = np.inf      # +inf: bad only when T > 0
    logits[3, 0, :100] = -np.inf  # masked vocabulary: fine
    draft[4, 1] = V               # invalid draft token
    dlen = np.full(B, K, np.int32)
    dlen[5] = K + 1               # invalid draft length
    for T in (0.0, 1.0):
        g, o, te, de = _run_both(ss, cuda_device, logits, draft, dlen, T=T)
        _check(g, o, te, de, draft, dlen, T)
        assert g["status"][0] == 5 and g["status"][1] == 5
        assert g["status"][4] == 6 and g["status"][5] == 6
        assert g["status"][3] == 0
        assert g["status"][2] == (5 if T > 0 else 0)


@pytest.mark.parametrize("with_draft", [False, True])
def test_malformed_rows_in_clusters(ss, cuda_device, with_draft):
    """The same malformed rows at the full vocabulary and B=8, where a
    sequence's fp32 tiles are shared by a cluster of CTAs and the tile's last
    warp merges its records: the NaN, the +inf and the only finite logit sit
    in tiles that the cluster's other CTAs stream (tile 1: logits 12288 up
    with fp32 rows, 6144 up with draft logits as well)."""
    B, K, V = 8, 2, workloads.V_LARGE
    logits, draft = workloads.sweep_host(510, B, K, V)
    rng = np.random.default_rng(511)
    tile1 = 6144 if with_draft else 12288
    draft[:] = np.argmax(logits[:, :K], axis=-1).astype(np.int32)
    logits[0, 0, tile1 + 17] = np.nan
    logits[1, 0, :] = -np.inf
    logits[2, 0, tile1 + 3] = np.inf     # +inf: bad only when T > 0
    logits[3, 0, :100] = -np.inf         # masked vocabulary: fine
    logits[4, 0, :] = -np.inf            # only the draft token finite
    draft[4, 0] = tile1 + 40
    logits[4, 0, tile1 + 40] = 1.5
    dl = None
    if with_draft:
        dl = (logits[:, :K] + workloads.gaussian_logits(rng, (B, K, V), 1.0)).astype(np.float32)
        dl[np.isnan(dl) | np.isinf(dl)] = 0.0
    for T in ((0.0, 1.0) if not with_draft else (1.0,)):
        g, o, te, de = _run_both(ss, cuda_device, logits, draft, None, T=T, seed=3,
                                 draft_logits=dl)
        _check(g, o, te, de, draft, None, T)
        assert g["status"][0] == 5 and g["status"][1] == 5
        assert g["status"][3] == 0 and g["status"][4] == 0 and g["accept_len"][4] >= 1
        assert g["status"][2] == (5 if T > 0 else 0)


def test_determinism_and_single_sequence(ss, cuda_device):
    B, K, V = 1, 3, 151936
    logits, draft = workloads.sweep_host(600, B, K, V)
    r1 = _run_both(ss, cuda_device, logits, draft, None, T=1.0, seed=9, step=4)[0]
    r2 = _run_both(ss, cuda_device, logits, draft, None, T=1.0, seed=9, step=4)[0]
    for k in ("accept_len", "out_token", "row_z", "p_d"):
        np.testing.assert_array_equal(r1[k], r2[k])


# points where the oracle checks every one of the 1024 sequences
FULL_POINTS = {(3, torch.bfloat16, 1.0), (3, torch.float32, 1.0), (8, torch.float32, 0.0),
               (1, torch.bfloat16, 0.0)}


@pytest.mark.parametrize("K", [1, 3, 5, 8])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("T", [0.0, 1.0])
def test_sweep_b1024_full_size(ss, cuda_device, K, dtype, T):
    """B=1024, V=151936 at full size in the benchmark's launch configuration.
    At four points the oracle verifies every sequence (rows copied back 128
    sequences at a time, the coins keyed by each sequence's index); at the
    others 24 sampled sequences."""
    B, V = 1024, 151936
    logits, draft = workloads.sweep_device(7000 + K, B, K, V, dtype, cuda_device)
    res = ss.spec_verify(logits, draft, None, temperature=T, seed=77, step=K, debug=True)
    g = gpu_to_numpy(res)
    assert (g["status"] == 0).all()
    dr_all = draft.cpu().numpy()
    if (K, dtype, T) in FULL_POINTS:
        chunks = [np.arange(b0, min(B, b0 + 128)) for b0 in range(0, B, 128)]
    else:
        chunks = [np.unique(np.concatenate([np.arange(0, B, 97), [B - 1]]))[:24]]
    decisions = excused = 0
    for sample in chunks:
        rows = logits[torch.as_tensor(sample, device=cuda_device)].float().cpu().numpy()
        dr = dr_all[sample]
        o = oracle.verify(rows, dr, None, temperature=T, seed=77, step=K, seq_index=sample)
        gs = {k: v[sample] for k, v in g.items()}
        d, e = compare_verify(gs, o, lambda i: rows[i], dr, None, T, budget=False)
        decisions += d
        excused += e
    assert excused <= int(1e-4 * decisions), f"{excused} excused of {decisions}"
    # acceptance is low (drafts uniform among the top-5): most sequences stop early
    assert (g["accept_len"] <= K).all()


@pytest.mark.parametrize("dtype,V,with_draft", [(torch.bfloat16, 48 * 24576, False),
                                                (torch.float32, 48 * 12288, False),
                                                (torch.float32, 32 * 6144, True)])
def test_largest_vocabulary(ss, cuda_device, dtype, V, with_draft):
    """The largest V each logits layout accepts (48 staging tiles with one-hot
    drafts, 32 with draft logits), and one more, which is refused."""
    B, K = 2, 1
    rng = np.random.default_rng(V)
    logits = workloads.gaussian_logits(rng, (B, K + 1, V), 2.0)
    draft = np.argsort(-logits[:, :K], axis=-1)[..., 3].astype(np.int32)
    dlog = None
    if with_draft:
        dlog = (logits[:, :K] + workloads.gaussian_logits(rng, (B, K, V), 1.0)).astype(np.float32)
    for T in (0.0, 1.0):
        g, o, te, de = _run_both(ss, cuda_device, logits, draft, None, T=T, seed=3,
                                 draft_logits=dlog if T > 0 else None, t_dtype=dtype)
        _check(g, o, te, de, draft, None, T)
    big = torch.zeros((1, K + 1, V + 64), dtype=dtype, device=cuda_device)
    with pytest.raises(ss.SamspecError):
        ss.spec_verify(big, torch.zeros((1, K), dtype=torch.int32, device=cuda_device), None,
                       temperature=1.0,
                       draft_logits=(torch.zeros((1, K, V + 64), dtype=torch.float32, device=cuda_device)
                                     if with_draft else None))


def test_only_the_draft_is_finite(ss, cuda_device):
    """A row whose only finite logit is the draft token: p is one-hot on it, so
    the draft is accepted (the sums without the draft are empty)."""
    B, K, V = 4, 2, 1000
    rng = np.random.default_rng(31)
    logits = workloads.gaussian_logits(rng, (B, K + 1, V), 2.0)
    draft = np.argsort(-logits[:, :K], axis=-1)[..., 2].astype(np.int32)
    for b in range(B):
        logits[b, 0, :] = -np.inf
        logits[b, 0, draft[b, 0]] = 1.5
    for T in (0.0, 1.0):
        g, o, te, de = _run_both(ss, cuda_device, logits, draft, None, T=T, seed=2)
        _check(g, o, te, de, draft, None, T)
        assert (g["status"] == 0).all() and (g["accept_len"] >= 1).all()
