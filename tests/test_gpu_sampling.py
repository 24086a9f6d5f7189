"""Per-request temperature / top-k / top-p on the GPU against the oracle and
the definitions: the cut of every row (top-k exactly; top-p exactly, or
within 1e-6 of top_p in mass when the fixed-point sums put it on the other
side), and verification decisions identical except where a coin falls within
1e-6 of its threshold or CDF boundary (at most 1e-4 of the decisions)."""
import numpy as np
import pytest
import torch
from scipy import stats

import oracle
import workloads
from parity import BAND, compare_sampling, cut_ok

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ss(cuda_device):
    import sam_drafting_verification_gb300 as ss
    return ss


def _params(rng, B, V):
    T = rng.choice([0.4, 0.7, 1.0, 1.7], B).astype(np.float32)
    k = rng.choice([-1, 0, 1, 5, 50, 1000, V, V + 3], B).astype(np.int32)
    p = rng.choice([0.1, 0.5, 0.9, 0.99, 1.0, 1.2], B).astype(np.float32)
    return T, k, p


@pytest.mark.parametrize("dtype,V", [(torch.float32, 3000), (torch.bfloat16, 40000),
                                     (torch.bfloat16, 40001), (torch.float32, 2999)])
def test_cut_matches_oracle(ss, cuda_device, dtype, V):
    rng = np.random.default_rng(V)
    B, R = 48, 3
    logits = workloads.gaussian_logits(rng, (B, R, V), 2.0)
    if dtype == torch.float32:
        logits[::3] = np.round(logits[::3] * 4) / 4  # many exact ties
    tl = torch.from_numpy(logits).to(dtype)
    rows = tl.float().numpy()
    T, k, p = _params(rng, B, V)
    dev = cuda_device
    tau = ss.sampling_cut(tl.to(dev), torch.from_numpy(T).to(dev), torch.from_numpy(k).to(dev),
                          torch.from_numpy(p).to(dev)).cpu().numpy()
    excused = 0
    for b in range(B):
        for r in range(R):
            if not (0 < k[b] < V) and not (p[b] < 1.0):
                assert tau[b, r] == -np.inf
                continue
            _, to = oracle.truncate_row(rows[b, r], float(T[b]), int(k[b]), float(p[b]))
            ok, ex = cut_ok(rows[b, r], float(T[b]), int(k[b]), float(p[b]), float(tau[b, r]), to)
            assert ok, (b, r, T[b], k[b], p[b], tau[b, r], to)
            excused += ex
    assert excused <= int(1e-4 * B * R), excused


def test_cut_bad_parameters_and_rows(ss, cuda_device):
    B, R, V = 6, 2, 64
    logits = torch.randn((B, R, V), device=cuda_device)
    logits[5, 1, 3] = float("nan")
    T = torch.tensor([0.0, float("inf"), float("nan"), 1.0, 1.0, 1.0], device=cuda_device)
    p = torch.tensor([0.9, 0.9, 0.9, 0.0, float("nan"), 0.9], device=cuda_device)
    tau = ss.sampling_cut(logits, T, 5, p).cpu().numpy()
    assert np.isnan(tau[:5]).all()
    assert np.isfinite(tau[5, 0]) and tau[5, 1] == -np.inf


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_verify_sampling_matches_oracle(ss, cuda_device, dtype):
    rng = np.random.default_rng(11 if dtype == torch.float32 else 12)
    B, K, V = 96, 3, 30000
    logits = workloads.gaussian_logits(rng, (B, K + 1, V), 2.0)
    top = np.argsort(-logits[:, :K], axis=-1)[..., :5]
    draft = np.take_along_axis(top, rng.integers(0, 5, (B, K, 1)), -1)[..., 0].astype(np.int32)
    tl = torch.from_numpy(logits).to(dtype)
    rows = tl.float().numpy()
    T, k, p = _params(rng, B, V)
    dev = cuda_device
    args = [torch.from_numpy(a).to(dev) for a in (T, k, p)]
    g = ss.spec_verify_sampling(tl.to(dev), torch.from_numpy(draft).to(dev), None, *args,
                                seed=17, step=5, emit=True)
    g = {key: v.cpu().numpy() for key, v in g.items()}
    tau_g = ss.sampling_cut(tl.to(dev), *args).cpu().numpy()
    o = oracle.verify_sampling(rows, draft, None, T, k, p, seed=17, step=5)
    compare_sampling(g, o, rows, draft, T, k, p, tau_g)
    assert (g["accept_len"] > 0).any()
    # emitted tokens: the accepted drafts, then the final token
    for b in range(B):
        L = g["accept_len"][b]
        assert list(g["emit"][b, :L + 1]) == list(draft[b, :L]) + [g["out_token"][b]]


def test_no_truncation_equals_spec_verify(ss, cuda_device):
    rng = np.random.default_rng(21)
    B, K, V = 64, 4, 20000
    for dtype in (torch.float32, torch.bfloat16):
        logits = torch.from_numpy(workloads.gaussian_logits(rng, (B, K + 1, V), 2.0)).to(dtype).to(cuda_device)
        draft = torch.argsort(logits[:, :K].float(), dim=-1, descending=True)[..., 1].to(torch.int32).contiguous()
        for T in (0.6, 1.0):
            a = ss.spec_verify(logits, draft, None, temperature=T, seed=3, step=1, emit=True)
            s = ss.spec_verify_sampling(logits, draft, None, T, 0, 1.0, seed=3, step=1, emit=True)
            for key in ("accept_len", "out_token", "emit", "status"):
                assert torch.equal(a[key], s[key]), key


def test_top1_equals_greedy(ss, cuda_device):
    rng = np.random.default_rng(22)
    B, K, V = 64, 4, 20000
    logits = torch.from_numpy(workloads.gaussian_logits(rng, (B, K + 1, V), 2.0)).to(cuda_device)
    am = torch.argmax(logits[:, :K], dim=-1).to(torch.int32)
    draft = torch.where(torch.rand((B, K), device=cuda_device) < 0.7, am, (am + 1) % V).contiguous()
    gr = ss.spec_verify(logits, draft, None, temperature=0.0)
    for T in (0.3, 2.0):
        s = ss.spec_verify_sampling(logits, draft, None, T, 1, 1.0, seed=5)
        assert torch.equal(gr["accept_len"], s["accept_len"])
        assert torch.equal(gr["out_token"], s["out_token"])


def test_first_token_follows_the_truncated_distribution(ss, cuda_device):
    """Losslessness on the device: identical rows, coins differing by
    sequence; the first emitted token's frequencies follow p'."""
    rng = np.random.default_rng(23)
    V, B, T, k, p = 16, 200000, 0.8, 9, 0.9
    row = workloads.gaussian_logits(rng, (V,), 1.0)
    logits = torch.from_numpy(np.stack([row, row])).to(cuda_device).expand(B, 2, V).contiguous()
    d = int(np.argsort(-row)[2])
    draft = torch.full((B, 1), d, dtype=torch.int32, device=cuda_device)
    g = ss.spec_verify_sampling(logits, draft, None, T, k, p, seed=29, step=0)
    assert (g["status"] == 0).all()
    first = torch.where(g["accept_len"] >= 1, draft[:, 0], g["out_token"]).cpu().numpy()
    pp, tau = oracle.truncate_row(row, T, k, p)
    counts = np.bincount(first, minlength=V)
    keep = pp > 0
    assert (counts[~keep] == 0).all()
    assert stats.chisquare(counts[keep], pp[keep] * B).pvalue > 1e-3


def test_bad_parameters(ss, cuda_device):
    B, K, V = 6, 2, 100
    logits = torch.randn((B, K + 1, V), device=cuda_device)
    draft = torch.zeros((B, K), dtype=torch.int32, device=cuda_device)
    T = torch.tensor([0.0, float("inf"), float("nan"), 1.0, 1.0, 1.0], device=cuda_device)
    p = torch.tensor([0.9, 0.9, 0.9, 0.0, float("nan"), 0.9], device=cuda_device)
    g = ss.spec_verify_sampling(logits, draft, None, T, 5, p)
    assert g["status"].cpu().tolist() == [8, 8, 8, 8, 8, 0]
    assert (g["accept_len"][:5] == -1).all()


def _check_cuts(ss, dev, rows_bf16, T, k, p):
    """Cuts of bf16 rows [B, R, V] against the oracle; returns the number of
    excused top-p boundary rows."""
    tl = torch.from_numpy(rows_bf16.astype(np.float32)).to(torch.bfloat16)
    rows = tl.float().numpy()
    B, R, V = rows.shape
    tau = ss.sampling_cut(tl.to(dev), torch.from_numpy(T).to(dev), torch.from_numpy(k).to(dev),
                          torch.from_numpy(p).to(dev)).cpu().numpy()
    excused = 0
    for b in range(B):
        for r in range(R):
            if not (0 < k[b] < V) and not (p[b] < 1.0):  # no truncation: nothing cut
                assert tau[b, r] == -np.inf, (b, r)
                continue
            res = oracle.truncate_row(rows[b, r], float(T[b]), int(k[b]), float(p[b]))
            if res is None:  # a row the verifier refuses
                assert tau[b, r] == -np.inf, (b, r)
                continue
            ok, ex = cut_ok(rows[b, r], float(T[b]), int(k[b]), float(p[b]), float(tau[b, r]), res[1])
            assert ok, (b, r, T[b], k[b], p[b], tau[b, r], res[1])
            excused += ex
    return excused


def test_cut_bf16_signed_zeros_infinities_and_ties(ss, cuda_device):
    """Rows whose cut falls among +0 and -0 (equal values on both sides of the
    sign), rows with -inf logits (counted by top-k, massless for top-p), rows
    of few distinct values, and refused rows (NaN, +inf, only -inf)."""
    rng = np.random.default_rng(31)
    V = 4096
    base = []
    zeros = np.zeros(V, np.float32)
    zeros[: V // 2] = -0.0
    zeros[rng.choice(V, 12, replace=False)] = rng.uniform(0.5, 2.0, 12)
    base.append(zeros)
    ninf = workloads.gaussian_logits(rng, (V,), 2.0)
    ninf[rng.choice(V, V - 30, replace=False)] = -np.inf
    base.append(ninf)
    few = rng.choice(np.array([-1.0, 0.0, 0.5, 1.0, 3.0], np.float32), V)
    base.append(few)
    mixed = workloads.gaussian_logits(rng, (V,), 2.0)
    mixed[rng.choice(V, 200, replace=False)] = -np.inf
    mixed[rng.choice(V, 300, replace=False)] = 0.0
    mixed[rng.choice(V, 300, replace=False)] = -0.0
    base.append(mixed)
    params = [(1.0, 5, 1.0), (1.0, 13, 1.0), (0.7, 0, 0.5), (1.0, 40, 0.95), (2.0, 0, 0.999),
              (1.0, 1000, 1.0), (0.5, 2500, 0.9)]
    rows = np.stack([np.stack(base)] * len(params))  # [P, 4, V]
    T = np.array([q[0] for q in params], np.float32)
    k = np.array([q[1] for q in params], np.int32)
    p = np.array([q[2] for q in params], np.float32)
    assert _check_cuts(ss, cuda_device, rows, T, k, p) <= 2
    bad = workloads.gaussian_logits(rng, (3, 1, V), 2.0)
    bad[0, 0, 7] = np.nan
    bad[1, 0, 9] = np.inf
    bad[2, 0, :] = -np.inf
    ones = np.ones(3, np.float32)
    tau = ss.sampling_cut(torch.from_numpy(bad).to(torch.bfloat16).to(cuda_device),
                          torch.from_numpy(ones).to(cuda_device), 5, 0.9).cpu().numpy()
    assert (tau == -np.inf).all()


@pytest.mark.parametrize("value", [1.0, 1.0078125, -np.inf])
def test_cut_bf16_many_equal_logits(ss, cuda_device, value):
    """More than 65,535 logits of one value (bf16 patterns of both parities,
    and -inf) take the radix path; 65,535 exactly does not.  Both agree with
    the oracle."""
    rng = np.random.default_rng(32)
    V = 151936
    rows = workloads.gaussian_logits(rng, (3, 2, V), 2.0)
    for i, n in enumerate((65535, 65536, 120000)):
        for r in range(2):
            rows[i, r, rng.choice(V, n, replace=False)] = value
    T = np.array([1.0, 0.8, 1.0], np.float32)
    k = np.array([50, 0, 70000], np.int32)
    p = np.array([0.9, 0.95, 1.0], np.float32)
    assert _check_cuts(ss, cuda_device, rows, T, k, p) == 0
    const = np.full((2, 1, V), value if np.isfinite(value) else 0.5, np.float32)
    assert _check_cuts(ss, cuda_device, const, np.ones(2, np.float32), np.array([10, 0], np.int32),
                       np.array([0.5, 0.3], np.float32)) == 0


def test_cut_full_vocab_sampled(ss, cuda_device):
    """The benchmark's shape (V = 151936 bf16, 4 rows per sequence, mixed
    parameters, more rows than SMs): every row cut on the device, 24 sampled
    rows checked against the oracle."""
    rng = np.random.default_rng(33)
    B, R, V = 96, 4, 151936
    logits = workloads.gaussian_logits(rng, (B, R, V), 2.0)
    tl = torch.from_numpy(logits).to(torch.bfloat16)
    rows = tl.float().numpy()
    T = rng.choice([0.6, 0.8, 1.0], B).astype(np.float32)
    k = rng.choice([0, 20, 50], B).astype(np.int32)
    p = rng.choice([0.9, 0.95, 1.0], B).astype(np.float32)
    dev = cuda_device
    tau = ss.sampling_cut(tl.to(dev), torch.from_numpy(T).to(dev), torch.from_numpy(k).to(dev),
                          torch.from_numpy(p).to(dev)).cpu().numpy()
    excused = 0
    for i in rng.choice(B * R, 24, replace=False):
        b, r = divmod(int(i), R)
        if k[b] == 0 and p[b] >= 1.0:
            assert tau[b, r] == -np.inf
            continue
        _, to = oracle.truncate_row(rows[b, r], float(T[b]), int(k[b]), float(p[b]))
        ok, ex = cut_ok(rows[b, r], float(T[b]), int(k[b]), float(p[b]), float(tau[b, r]), to)
        assert ok, (b, r, tau[b, r], to)
        excused += ex
    assert excused == 0


@pytest.mark.parametrize("V", [1, 2, 7, 8, 9])
def test_cut_bf16_tiny_vocabularies(ss, cuda_device, V):
    """Vocabularies of a few logits (row lengths that are and are not whole
    16-byte vectors), with ties, against the oracle."""
    rng = np.random.default_rng(50 + V)
    rows = np.round(workloads.gaussian_logits(rng, (6, 2, V), 2.0) * 2) / 2
    T = np.array([1.0, 0.5, 2.0, 1.0, 0.7, 1.0], np.float32)
    k = np.array([1, 2, 0, 3, 1, 0], np.int32)
    p = np.array([1.0, 0.9, 0.5, 0.3, 0.99, 0.01], np.float32)
    assert _check_cuts(ss, cuda_device, rows, T, k, p) == 0
