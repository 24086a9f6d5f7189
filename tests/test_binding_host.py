"""Host logic of the Python binding (no GPU): every tensor it hands to the C
ABI is checked first -- inputs, the caller's output buffers and workspaces
alike -- and a rejected call reaches no entry point.  The library is replaced
by a recorder and the CUDA-tensor test by one that accepts host tensors, so
only the binding's own checks and argument marshalling run."""
import pytest
import torch

import sam_drafting_verification_gb300 as ss

B, K, V = 4, 3, 64


class _Recorder:
    """Stands in for libsamspec.so: records each entry point called."""

    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        def entry(*args):
            self.calls.append((name, args))
            return 0
        return entry


@pytest.fixture
def lib(monkeypatch):
    rec = _Recorder()
    monkeypatch.setattr(ss._b, "lib", lambda: rec)
    monkeypatch.setattr(ss, "_is_cuda", lambda t: t.device.type in ("cpu", "meta"))
    monkeypatch.setattr(ss, "_stream", lambda device=None: None)
    return rec


def _i32(*shape):
    return torch.zeros(shape, dtype=torch.int32)


def _verify_args():
    target = torch.zeros((B, K + 1, V), dtype=torch.bfloat16)
    return target, _i32(B, K), torch.zeros(256, dtype=torch.uint8)


def _ptr_value(p):
    return None if p is None else p.value


def test_valid_call_reuses_the_callers_buffers(lib):
    target, draft, ws = _verify_args()
    out = {"accept_len": _i32(B), "out_token": _i32(B), "status": _i32(B), "emit": _i32(B, K + 1),
           "emit_len": _i32(B)}
    res = ss.spec_verify(target, draft, temperature=1.0, out=out, emit=True, workspace=ws)
    assert res is out
    (name, args), = lib.calls
    assert name == "spec_verify"
    passed = {_ptr_value(a) for a in args if hasattr(a, "value")}
    for t in list(out.values()) + [target, draft, ws]:
        assert t.data_ptr() in passed


@pytest.mark.parametrize("key,bad,err", [
    ("accept_len", torch.zeros(B, dtype=torch.float32), TypeError),
    ("out_token", torch.zeros(B + 1, dtype=torch.int32), ValueError),
    ("status", torch.zeros(B, dtype=torch.int64), TypeError),
    ("emit", torch.zeros((K + 1, B), dtype=torch.int32).t(), ValueError),   # not contiguous
    ("emit_len", torch.zeros(B, dtype=torch.int32, device="meta"), ValueError),  # another device
])
def test_bad_output_buffer_is_refused_before_any_call(lib, key, bad, err):
    target, draft, ws = _verify_args()
    out = {key: bad}
    with pytest.raises(err, match=r"out\[" + key + r"\]"):
        ss.spec_verify(target, draft, temperature=1.0, out=out, emit=True, workspace=ws)
    assert lib.calls == []


def test_a_passed_buffer_is_checked_even_when_not_requested(lib):
    # an emit buffer in `out` is handed to the kernel whatever `emit` says
    target, draft, ws = _verify_args()
    with pytest.raises(ValueError, match=r"out\[emit\]"):
        ss.spec_verify(target, draft, out={"emit": _i32(B, K)}, emit=False, workspace=ws)
    assert lib.calls == []


@pytest.mark.parametrize("bad,err", [
    (torch.zeros(64, dtype=torch.int32), TypeError),
    (torch.zeros(256, dtype=torch.uint8, device="meta"), ValueError),
    (torch.zeros((16, 32), dtype=torch.uint8).t(), ValueError),
])
def test_bad_workspace_is_refused(lib, bad, err):
    target, draft, _ = _verify_args()
    with pytest.raises(err, match="workspace"):
        ss.spec_verify(target, draft, workspace=bad)
    assert lib.calls == []


@pytest.mark.parametrize("what", ["draft_device", "draft_len_shape", "draft_logits_dtype"])
def test_bad_inputs_are_refused(lib, what):
    target, draft, ws = _verify_args()
    kw = {}
    if what == "draft_device":
        draft = _i32(B, K).to("meta")
    elif what == "draft_len_shape":
        kw["draft_len"] = _i32(B, 1)
    else:
        kw["draft_logits"] = torch.zeros((B, K, V), dtype=torch.float16)
    with pytest.raises((TypeError, ValueError)):
        ss.spec_verify(target, draft, workspace=ws, temperature=1.0, **kw)
    assert lib.calls == []


def test_tree_outputs_checked_and_completed(lib):
    N = 4
    target = torch.zeros((B, N, V), dtype=torch.float32)
    tok, fc, ns = _i32(B, N), _i32(B, N), _i32(B, N)
    ws = torch.zeros(256, dtype=torch.uint8)
    with pytest.raises(ValueError, match=r"out\[path\]"):
        ss.spec_verify_tree(target, tok, fc, ns, workspace=ws, out={"path": _i32(B, N + 1)})
    assert lib.calls == []
    res = ss.spec_verify_tree(target, tok, fc, ns, workspace=ws, out={"path": _i32(B, N)})
    assert set(res) == {"accept_len", "out_token", "path", "emit", "emit_len", "status"}
    assert [c[0] for c in lib.calls] == ["spec_verify_tree"]


def test_sampling_parameters_and_outputs_checked(lib):
    target, draft, ws = _verify_args()
    with pytest.raises(ValueError, match="temperature"):
        ss.spec_verify_sampling(target, draft, temperature=torch.ones(B + 1), workspace=ws)
    with pytest.raises(TypeError, match=r"out\[emit_len\]"):
        ss.spec_verify_sampling(target, draft, workspace=ws, emit=True,
                                out={"emit_len": torch.zeros(B, dtype=torch.int64)})
    with pytest.raises(ValueError, match="top_k"):
        ss.sampling_cut(target, 1.0, _i32(B).to("meta"), 1.0)
    assert lib.calls == []
    ss.spec_verify_sampling(target, draft, temperature=torch.full((B,), 0.7), top_k=20, top_p=0.9,
                            workspace=ws)
    assert [c[0] for c in lib.calls] == ["spec_verify_sampling"]


def test_select_drafts_shapes_checked(lib):
    dyn = (_i32(B, K), _i32(B), _i32(B))
    with pytest.raises(ValueError, match="static draft"):
        ss.select_drafts(dyn, (_i32(B, K + 1), _i32(B), _i32(B)), 2)
    with pytest.raises(ValueError, match="static match_len"):
        ss.select_drafts(dyn, (_i32(B, K), _i32(B), _i32(B + 1)), 2)
    assert lib.calls == []
    ss.select_drafts(dyn, (_i32(B, K), _i32(B), _i32(B)), 2)
    assert [c[0] for c in lib.calls] == ["sam_select_drafts"]
