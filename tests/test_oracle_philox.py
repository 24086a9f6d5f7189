"""Pins of the oracle's Philox4x32-10 (no GPU).

The pages draw their coins with torch.rand; the reproducible coins here come
from Philox4x32-10 (Salmon et al., SC'11).  The oracle's implementation is
checked bit for bit against an independent third-party implementation, the
one in Triton's language library, run by Triton's CPU interpreter in a child
process, both for raw counters and for the counter layout of the coins;
the uniform map is checked at its end points and for uniformity.
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
from scipy import stats

import oracle

_TRITON_SCRIPT = r"""
import os, sys, json
os.environ["TRITON_INTERPRET"] = "1"
import numpy as np, torch, triton, triton.language as tl
from triton.language.random import philox

@triton.jit
def k(out_ptr, seed, c0p, c1p, c2p, c3p, N: tl.constexpr):
    i = tl.arange(0, N)
    a, b, c, d = philox(seed, tl.load(c0p + i), tl.load(c1p + i), tl.load(c2p + i), tl.load(c3p + i), 10)
    tl.store(out_ptr + i * 4 + 0, a)
    tl.store(out_ptr + i * 4 + 1, b)
    tl.store(out_ptr + i * 4 + 2, c)
    tl.store(out_ptr + i * 4 + 3, d)

req = json.loads(sys.stdin.read())
res = []
for seed, ctrs in req:
    C = np.array(ctrs, dtype=np.uint64).astype(np.uint32).T.copy()
    N = C.shape[1]
    out = torch.zeros(N * 4, dtype=torch.uint32)
    k[(1,)](out, seed, *[torch.from_numpy(C[i].copy()) for i in range(4)], N=N)
    res.append(out.view(N, 4).numpy().astype(np.int64).tolist())
print(json.dumps(res))
"""


def _triton_philox(req):
    """Philox4x32-10 words from Triton's library for [(seed, [counter, ...])]."""
    pytest.importorskip("triton")
    p = subprocess.run([sys.executable, "-c", _TRITON_SCRIPT], input=json.dumps(req),
                       capture_output=True, text=True, timeout=600,
                       env={**os.environ, "TRITON_INTERPRET": "1"})
    if p.returncode != 0:
        pytest.skip("triton interpreter unavailable: " + p.stderr.strip().splitlines()[-1][:200])
    return json.loads(p.stdout.strip().splitlines()[-1])


def test_philox_matches_triton_library():
    rng = np.random.default_rng(41)
    req = []
    seeds = [0, 1, 0xFFFFFFFF, 0x123456789ABCDEF, 2**64 - 1]
    for seed in seeds:
        ctrs = rng.integers(0, 2**32, size=(16, 4), dtype=np.uint64)
        ctrs[0] = 0
        ctrs[1] = 2**32 - 1
        req.append([seed, ctrs.tolist()])
    got = _triton_philox(req)
    for (seed, ctrs), tri in zip(req, got):
        key = [seed & 0xFFFFFFFF, seed >> 32]
        for c, t in zip(ctrs, tri):
            assert list(oracle.philox4x32_10(c, key)) == t, (seed, c)


def test_coin_counter_layout_matches_triton_library():
    # The coins of sequence b at draft position j in decoding step `step`:
    # key = (seed lo, seed hi), counter = (j, b, step lo, step hi); word 0
    # gives the accept coin u_j and word 1 the resample coin u'_j, each through
    # U(x) = ((x >> 9) + 1/2) * 2^-23.  Positions, sequences and steps are
    # chosen with distinct values so that a transposed counter word shows.
    cases = [(7, 3, 5, 2), (2**40 + 9, 2**33 + 17, 1000, 7), (0, 0, 0, 0), (12345, 1, 2**31 + 5, 31)]
    req = [[seed, [[j, b, step & 0xFFFFFFFF, step >> 32]]] for seed, step, b, j in cases]
    got = _triton_philox(req)
    for (seed, step, b, j), tri in zip(cases, got):
        w = tri[0]
        want = [((w[i] >> 9) + 0.5) * 2.0**-23 for i in (0, 1)]
        assert list(oracle.uniforms(seed, step, b, j)) == want, (seed, step, b, j)


def test_uniform_map_end_points_and_exactness():
    # U(x) = ((x >> 9) + 0.5) * 2^-23 lies strictly inside (0, 1) and is exact
    # in binary32: check through the oracle's uniforms over many counters.
    us = np.array([oracle.uniforms(77, s, b, j) for s in range(4) for b in range(64) for j in range(4)])
    assert np.all(us > 0) and np.all(us < 1)
    assert np.all(us.astype(np.float32).astype(np.float64) == us)
    k = us * 2**24
    assert np.all(k == np.round(k)) and np.all(np.round(k) % 2 == 1)


def test_uniforms_are_uniform_and_independent():
    us = np.array([oracle.uniforms(2024, s, b, j) for s in range(20) for b in range(250) for j in range(4)])
    for col in range(2):
        assert stats.kstest(us[:, col], "uniform").pvalue > 1e-3
    r = np.corrcoef(us[:, 0], us[:, 1])[0, 1]
    assert abs(r) < 4.0 / np.sqrt(len(us))
    # neighbouring counters decorrelated
    u0 = us[:-1, 0]
    u1 = us[1:, 0]
    assert abs(np.corrcoef(u0, u1)[0, 1]) < 4.0 / np.sqrt(len(u0))
