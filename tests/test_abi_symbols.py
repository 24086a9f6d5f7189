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


def test_binding_refuses_missing_library(tmp_path):
    import sam_drafting_verification_gb300._binding as bd
    with pytest.raises(bd.SamspecError):
        bd.load(str(tmp_path / "nope.so"))
