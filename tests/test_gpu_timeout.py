"""The verification kernels' bounded waits, made to run out on purpose.

With the wait limit shortened to a nanosecond through the library's test hook,
every on-chip wait that is not satisfied at once gives up: the kernel must
mark each sequence it did not finish with ST_TIMEOUT (accept_len and
out_token -1, emit_len 0), give every other sequence its full result, return,
and leave the context and the workspace usable -- the next call with the
default limit gives the reference results again.  Nothing here faults or
hangs the GPU: only the limit of the existing waits changes."""
import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

V = workloads.V_LARGE


def _lib():
    import sam_drafting_verification_gb300._binding as bd
    return bd, bd.lib()


def _outputs(B, K1, dev):
    o = {k: torch.full((B,), -7, dtype=torch.int32, device=dev)
         for k in ("accept_len", "out_token", "emit_len", "status")}
    o["emit"] = torch.full((B, K1), -7, dtype=torch.int32, device=dev)
    return o


def _check(ref, got, st_timeout):
    st = got["status"].cpu().numpy()
    timed = st == st_timeout
    assert timed.any(), "no wait ran out"
    assert ((st == 0) | timed).all(), np.unique(st)
    for k, v in (("accept_len", -1), ("out_token", -1), ("emit_len", 0)):
        assert (got[k].cpu().numpy()[timed] == v).all(), k
    assert (got["emit"].cpu().numpy()[timed] == -1).all()
    ok = ~timed
    for k in ("accept_len", "out_token", "emit_len", "emit"):
        assert np.array_equal(got[k].cpu().numpy()[ok], ref[k].cpu().numpy()[ok]), k
    return int(timed.sum())


@pytest.mark.parametrize("B,K,dtype,T", [(1024, 3, torch.bfloat16, 1.0), (1024, 3, torch.bfloat16, 0.0),
                                         (300, 5, torch.float32, 0.7), (8, 1, torch.bfloat16, 1.0)])
def test_expired_waits_mark_unfinished_sequences(cuda_device, B, K, dtype, T):
    import sam_drafting_verification_gb300 as ss
    bd, lib = _lib()
    logits, drafts = workloads.sweep_device(8100 + B + K, B, K, V, dtype, cuda_device)
    ws = torch.zeros(lib.spec_verify_workspace_bytes(B, K, V), dtype=torch.uint8, device=cuda_device)
    ref = ss.spec_verify(logits, drafts, temperature=T, seed=12, step=3, emit=True, status=True,
                         workspace=ws)
    torch.cuda.synchronize()
    assert (ref["status"] == 0).all()
    got = _outputs(B, K + 1, cuda_device)
    prev = lib.samspec_set_wait_limit_ns(1)
    try:
        ss.spec_verify(logits, drafts, temperature=T, seed=12, step=3, emit=True, status=True,
                       workspace=ws, out=got)
        torch.cuda.synchronize()
    finally:
        lib.samspec_set_wait_limit_ns(0)
    assert prev == 2_000_000_000
    n_timed = _check(ref, got, bd.ST_TIMEOUT)
    assert 0 < n_timed <= B
    # the context and the workspace are usable: the same call with the
    # default limit gives the reference results
    again = _outputs(B, K + 1, cuda_device)
    ss.spec_verify(logits, drafts, temperature=T, seed=12, step=3, emit=True, status=True,
                   workspace=ws, out=again)
    torch.cuda.synchronize()
    for k in ("accept_len", "out_token", "emit_len", "emit", "status"):
        assert torch.equal(again[k], ref[k]), k


def test_expired_waits_with_draft_logits_and_trees(cuda_device):
    import sam_drafting_verification_gb300 as ss
    bd, lib = _lib()
    w = workloads.draft_model(seed=8200, B=32, V=V, K=5)
    tgt = torch.as_tensor(w["target"], device=cuda_device)
    dl = torch.as_tensor(w["draft_logits"], device=cuda_device)
    dr = torch.as_tensor(w["draft"], device=cuda_device)
    ref = ss.spec_verify(tgt, dr, draft_logits=dl, temperature=0.7, seed=4, step=9, emit=True, status=True)
    torch.cuda.synchronize()
    got = _outputs(32, 6, cuda_device)
    lib.samspec_set_wait_limit_ns(1)
    try:
        ss.spec_verify(tgt, dr, draft_logits=dl, temperature=0.7, seed=4, step=9, emit=True, status=True,
                       out=got)
        torch.cuda.synchronize()
    finally:
        lib.samspec_set_wait_limit_ns(0)
    _check(ref, got, bd.ST_TIMEOUT)
    # a chain-shaped tree under the short limit: every sequence ends either
    # with the chain's result or with ST_TIMEOUT
    B, N = 48, 4
    rng = np.random.default_rng(8201)
    logits = torch.as_tensor(workloads.gaussian_logits(rng, (B, N, 40000), 2.0), device=cuda_device)
    tok = np.full((B, N), -1, np.int32)
    tok[:, 1:] = rng.integers(0, 40000, size=(B, N - 1))
    fc = np.tile(np.array([1, 2, 3, -1], np.int32), (B, 1))
    ns = np.full((B, N), -1, np.int32)
    args = [torch.as_tensor(a, device=cuda_device) for a in (tok, fc, ns)]
    tref = ss.spec_verify_tree(logits, *args, temperature=1.0, seed=2, step=1)
    torch.cuda.synchronize()
    lib.samspec_set_wait_limit_ns(1)
    try:
        tgot = ss.spec_verify_tree(logits, *args, temperature=1.0, seed=2, step=1)
        torch.cuda.synchronize()
    finally:
        lib.samspec_set_wait_limit_ns(0)
    st = tgot["status"].cpu().numpy()
    assert (st == bd.ST_TIMEOUT).any() and ((st == 0) | (st == bd.ST_TIMEOUT)).all()
    ok = st == 0
    for k in ("accept_len", "out_token", "path", "emit"):
        assert np.array_equal(tgot[k].cpu().numpy()[ok], tref[k].cpu().numpy()[ok]), k
    after = ss.spec_verify_tree(logits, *args, temperature=1.0, seed=2, step=1)
    for k in ("accept_len", "out_token", "path", "emit", "status"):
        assert torch.equal(after[k], tref[k]), k
