"""The C-ABI library loads without a GPU and exports every entry point that
include/samspec.h declares (no compute calls)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "samspec.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:[A-Za-z_][\w\s\*]*?)\b([a-z_][a-z0-9_]*)\s*\(", src, flags=re.M)
    return sorted({n for n in names if n not in ("if", "sizeof")})


def test_library_exports_every_declared_symbol():
    from sam_drafting_verification_gb300 import build as b
    path = b.build()
    lib = ctypes.CDLL(path)
    declared = _declared()
    assert len(declared) >= 15, declared
    missing = [n for n in declared if not hasattr(lib, n)]
    assert not missing, missing
    from sam_drafting_verification_gb300 import _binding
    assert sorted(_binding.EXPORTED) == declared


def test_host_only_calls():
    import sam_drafting_verification_gb300._binding as bd
    lib = bd.lib()
    assert lib.samspec_version() == 100
    assert lib.sam_batch_workspace_bytes(0, 10) == 0
    assert lib.sam_batch_workspace_bytes(1, 1 << 22) == 0
    assert lib.sam_batch_workspace_bytes(4, 256) > 0
    assert lib.spec_verify_workspace_bytes(4, 3, 100) >= 16
    assert lib.samspec_strerror(-1) == b"invalid argument"


def test_spec_verify_rejects_bad_arguments_on_the_host():
    """Argument checks return before any device work, so they run without a
    GPU: the pointers below are aligned placeholders that are never touched."""
    import sam_drafting_verification_gb300._binding as bd
    lib = bd.lib()
    p = ctypes.c_void_p(4096)

    def call(dtype=bd.F32, K=1, V=1000, T=1.0, ws_bytes=256, target=p, draft_logits=None):
        return lib.spec_verify(target, dtype, draft_logits, bd.F32, p, None, 1, K, V, T, 0, 0, p, p,
                               None, None, None, None, p, ws_bytes, None)

    assert call(target=None) == bd.EINVAL
    assert call(K=-1) == bd.ESIZE and call(K=33) == bd.ESIZE
    assert call(T=-1.0) == bd.EINVAL and call(T=float("nan")) == bd.EINVAL
    assert call(dtype=7) == bd.EDTYPE
    assert call(ws_bytes=16) == bd.ESIZE
    assert call(target=ctypes.c_void_p(4100)) == bd.EALIGN
    # V above 48 staging tiles: 12288 fp32 / 24576 bf16 logits per tile
    assert call(dtype=bd.F32, V=48 * 12288 + 1) == bd.ESIZE
    assert call(dtype=bd.BF16, V=48 * 24576 + 1) == bd.ESIZE
    assert call(dtype=bd.F32, V=48 * 12288 + 1, T=0.0) == bd.ESIZE
    # with draft logits (T > 0) both rows share a tile: 32 tiles of 6144 fp32 pairs
    assert call(dtype=bd.F32, V=32 * 6144 + 1, draft_logits=p, ws_bytes=1 << 20) == bd.ESIZE


def test_binding_refuses_missing_library(tmp_path):
    import sam_drafting_verification_gb300._binding as bd
    with pytest.raises(bd.SamspecError):
        bd.load(str(tmp_path / "nope.so"))


def test_sampling_entry_points_reject_bad_arguments_on_the_host():
    """Argument checks of spec_sampling_cut and spec_verify_sampling, which
    return before any device work (placeholders are never touched)."""
    import sam_drafting_verification_gb300._binding as bd
    lib = bd.lib()
    p = ctypes.c_void_p(4096)
    assert lib.spec_verify_sampling_workspace_bytes(4, 3, 100) >= 256 + 4 * 4 * 4
    assert lib.spec_verify_sampling_workspace_bytes(0, 3, 100) == 0

    def cut(target=p, dtype=bd.F32, B=2, R=2, V=100, temp=p):
        return lib.spec_sampling_cut(target, dtype, B, R, V, temp, p, p, p, None)

    assert cut(target=None) == bd.EINVAL and cut(temp=None) == bd.EINVAL
    assert cut(R=34) == bd.ESIZE and cut(V=(1 << 21) + 1) == bd.ESIZE and cut(B=0) == bd.ESIZE
    assert cut(dtype=9) == bd.EDTYPE
    assert cut(target=ctypes.c_void_p(4100)) == bd.EALIGN

    def ver(dtype=bd.BF16, K=2, V=1000, ws_bytes=1 << 16, draft=p, top_p=p):
        return lib.spec_verify_sampling(p, dtype, draft, None, 2, K, V, p, p, top_p, 0, 0, p, p,
                                        None, None, p, None, p, ws_bytes, None)

    assert ver(draft=None) == bd.EINVAL and ver(top_p=None) == bd.EINVAL
    assert ver(K=33) == bd.ESIZE and ver(ws_bytes=256) == bd.ESIZE
    assert ver(V=48 * 24576 + 1) == bd.ESIZE and ver(dtype=bd.F32, V=48 * 12288 + 1) == bd.ESIZE
    assert ver(dtype=5) == bd.EDTYPE


def test_strerror_names_every_code_the_header_defines():
    """Every return code and status word in include/samspec.h has its own text."""
    import sam_drafting_verification_gb300._binding as bd
    lib = bd.lib()
    src = open(os.path.join(ROOT, "include", "samspec.h")).read()
    codes = {m[0]: int(m[1]) for m in
             re.findall(r"#define\s+(SAMSPEC_(?:OK|E[A-Z]+|ST_[A-Z]+))\s+\(?(-?\d+)\)?", src)}
    assert {"SAMSPEC_OK", "SAMSPEC_EINVAL", "SAMSPEC_ST_TIMEOUT", "SAMSPEC_ST_BADPARAM"} <= set(codes)
    texts = {}
    for name, v in codes.items():
        t = lib.samspec_strerror(v)
        assert t != b"unknown code", name
        texts.setdefault(v, t)
    # return codes and status words share only 0 (ok)
    assert len(set(texts.values())) == len(texts)
    assert lib.samspec_strerror(12345) == b"unknown code"
