"""spec_verify_noalloc, the verification entry point for callers that cannot
allocate device memory (their runtime owns every allocation, or allocating
would synchronise the device), checked against spec_verify through the C ABI.

The file is named so that pytest collects it last: the entry point shares one
library-held scratch array per device, and the test must hold both in a fresh
process and after every other test has used the library."""
import ctypes

import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _outputs(B, K1, dev):
    o = {k: torch.full((B,), -7, dtype=torch.int32, device=dev)
         for k in ("accept_len", "out_token", "emit_len", "status")}
    o["emit"] = torch.full((B, K1), -7, dtype=torch.int32, device=dev)
    for k in ("row_m", "row_z", "p_d", "q_d"):
        o[k] = torch.full((B, K1), float("nan"), dtype=torch.float32, device=dev)
    o["row_arg"] = torch.full((B, K1), -1, dtype=torch.int32, device=dev)
    o["res_mass"] = torch.full((B,), float("nan"), dtype=torch.float32, device=dev)
    return o


def _call(bd, lib, noalloc, target, draft, T, seed, step, out, ws=None):
    B, K1, V = target.shape
    dt = bd.F32 if target.dtype == torch.float32 else bd.BF16
    dbg = bd.VerifyDebug(*[out[k].data_ptr() for k in ("row_m", "row_z", "p_d", "q_d", "row_arg", "res_mass")])
    stream = ctypes.c_void_p(torch.cuda.current_stream(target.device).cuda_stream)
    args = [_ptr(target), dt, None, bd.F32, _ptr(draft), None, B, K1 - 1, V, float(T), seed, step,
            _ptr(out["accept_len"]), _ptr(out["out_token"]), _ptr(out["emit"]), _ptr(out["emit_len"]),
            _ptr(out["status"]), ctypes.byref(dbg)]
    if noalloc:
        return lib.spec_verify_noalloc(*args, stream)
    return lib.spec_verify(*args, _ptr(ws), ws.numel(), stream)


def test_noalloc_matches_spec_verify_twice(cuda_device):
    import sam_drafting_verification_gb300._binding as bd
    lib = bd.lib()
    B, K, V = 96, 3, 50257
    logits, draft = workloads.sweep_host(4242, B, K, V)
    target = torch.from_numpy(logits).to(torch.bfloat16).to(cuda_device)
    drafts = torch.as_tensor(draft, device=cuda_device)
    ws = torch.zeros(lib.spec_verify_workspace_bytes(B, K, V), dtype=torch.uint8, device=cuda_device)
    # two calls in a row: sampling then greedy, each against spec_verify
    for T, step in ((1.0, 5), (0.0, 6)):
        ref = _outputs(B, K + 1, cuda_device)
        new = _outputs(B, K + 1, cuda_device)
        assert _call(bd, lib, False, target, drafts, T, 31, step, ref, ws) == bd.OK
        assert _call(bd, lib, True, target, drafts, T, 31, step, new) == bd.OK
        torch.cuda.synchronize(cuda_device)
        for k in ("accept_len", "out_token", "emit", "emit_len", "status", "row_arg"):
            assert torch.equal(new[k], ref[k]), k
        assert (new["status"] == 0).all()
        for k in ("row_m", "row_z", "p_d", "q_d", "res_mass"):
            a, b = new[k].cpu().numpy(), ref[k].cpu().numpy()
            assert np.array_equal(np.isnan(a), np.isnan(b)), k
            m = ~np.isnan(b)
            # the same kernel on the same inputs: within the 1e-6 relative
            # tolerance of the parity tests (in practice identical)
            assert (np.abs(a[m] - b[m]) <= 1e-6 * np.maximum(np.abs(b[m]), 1e-30)).all(), k


def test_noalloc_rejects_sizes_beyond_its_limits(cuda_device):
    import sam_drafting_verification_gb300._binding as bd
    lib = bd.lib()
    B, K, V = 4, 33, 1000  # K above the 32 drafts a call accepts
    target = torch.zeros((B, K + 1, V), dtype=torch.float32, device=cuda_device)
    drafts = torch.zeros((B, K), dtype=torch.int32, device=cuda_device)
    out = _outputs(B, K + 1, cuda_device)
    rc = _call(bd, lib, True, target, drafts, 1.0, 0, 0, out)
    assert rc == bd.ESIZE
    assert b"size" in lib.samspec_strerror(rc).lower()
    assert (out["accept_len"] == -7).all()  # nothing was launched
