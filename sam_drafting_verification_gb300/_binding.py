"""ctypes binding of libsamspec.so: argument marshalling only.

Every computation runs in the library's CUDA kernels; torch supplies device
memory and the current stream.  The in-tree library is loaded at the first
call that needs it; if it is missing, that call raises SamspecError (build it
with ``python -m sam_drafting_verification_gb300.build``): there is no
fallback.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libsamspec.so")
# the debug build: every automaton index checked against its array (ST_BOUNDS)
CHECKS_LIB_PATH = os.path.join(_HERE, "_lib", "libsamspec_checks.so")

# host-side return codes and per-sequence status words (include/samspec.h)
OK, EINVAL, ESIZE, EDTYPE, ECUDA, EALIGN = 0, -1, -2, -3, -4, -5
(ST_OK, ST_CAPACITY, ST_HASHFULL, ST_TOKEN, ST_LOOPCAP, ST_BADROW, ST_BADDRAFT, ST_TIMEOUT, ST_BADPARAM,
 ST_BOUNDS) = range(10)
F32, BF16 = 0, 1

EXPORTED = [
    "samspec_version", "samspec_strerror",
    "sam_batch_workspace_bytes", "sam_batch_create", "sam_batch_destroy", "sam_reset",
    "sam_extend", "sam_draft", "sam_step", "sam_get_status", "sam_export", "sam_import",
    "sam_dump_sequence",
    "spec_verify_workspace_bytes", "spec_verify_workspace_init", "spec_verify", "spec_uniforms",
    "spec_verify_noalloc", "sam_step_rows", "sam_spec_step", "ssam_match", "sam_select_drafts",
    "spec_verify_tree", "spec_sampling_cut", "spec_verify_sampling_workspace_bytes",
    "spec_verify_sampling", "samspec_set_wait_limit_ns",
]


class SamspecError(RuntimeError):
    pass


class VerifyDebug(ctypes.Structure):
    _fields_ = [("row_m", ctypes.c_void_p), ("row_z", ctypes.c_void_p), ("p_d", ctypes.c_void_p),
                ("q_d", ctypes.c_void_p), ("row_arg", ctypes.c_void_p), ("res_mass", ctypes.c_void_p)]


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise SamspecError(f"libsamspec.so not built at {path}; run "
                           "`python -m sam_drafting_verification_gb300.build`")
    lib = ctypes.CDLL(path)
    P, I32, U64, SZ, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint64, ctypes.c_size_t, ctypes.c_float
    sig = {
        "samspec_version": (ctypes.c_int, []),
        "samspec_strerror": (ctypes.c_char_p, [ctypes.c_int]),
        "sam_batch_workspace_bytes": (SZ, [I32, I32]),
        "sam_batch_create": (ctypes.c_int, [I32, I32, I32, P, SZ, P, ctypes.POINTER(P)]),
        "sam_batch_destroy": (ctypes.c_int, [P]),
        "sam_reset": (ctypes.c_int, [P, P, P]),
        "sam_extend": (ctypes.c_int, [P, P, P, I32, P]),
        "sam_draft": (ctypes.c_int, [P, I32, P, P, P, P, P]),
        "sam_step": (ctypes.c_int, [P, P, P, I32, I32, P, P, P, P, P]),
        "sam_get_status": (ctypes.c_int, [P, P, P]),
        "sam_export": (ctypes.c_int, [P, P, SZ, P]),
        "sam_import": (ctypes.c_int, [P, P, SZ, P]),
        "sam_dump_sequence": (ctypes.c_int, [P, I32, P, P, P, P, I32, P, I32, P]),
        "spec_verify_workspace_bytes": (SZ, [I32, I32, I32]),
        "spec_verify_workspace_init": (ctypes.c_int, [P, SZ, P]),
        "spec_verify": (ctypes.c_int, [P, I32, P, I32, P, P, I32, I32, I32, F, U64, U64,
                                       P, P, P, P, P, ctypes.POINTER(VerifyDebug), P, SZ, P]),
        "spec_uniforms": (ctypes.c_int, [I32, I32, U64, U64, P, P]),
        "samspec_set_wait_limit_ns": (U64, [U64]),
        "spec_verify_noalloc": (ctypes.c_int, [P, I32, P, I32, P, P, I32, I32, I32, F, U64, U64,
                                               P, P, P, P, P, ctypes.POINTER(VerifyDebug), P]),
        "sam_step_rows": (ctypes.c_int, [P, P, I32, P, P, I32, I32, P, P, P, P, P]),
        "ssam_match": (ctypes.c_int, [P, I32, I32, P, P, P, I32, I32, P, P, P, P, P]),
        "spec_verify_tree": (ctypes.c_int, [P, I32, P, P, P, I32, I32, I32, F, U64, U64, P, P, P,
                                            P, P, P, ctypes.POINTER(VerifyDebug), P, SZ, P]),
        "sam_select_drafts": (ctypes.c_int, [I32, I32, P, P, P, P, P, P, I32, P, P, P, P]),
        "spec_sampling_cut": (ctypes.c_int, [P, I32, I32, I32, I32, P, P, P, P, P]),
        "spec_verify_sampling_workspace_bytes": (SZ, [I32, I32, I32]),
        "spec_verify_sampling": (ctypes.c_int, [P, I32, P, P, I32, I32, I32, P, P, P, U64, U64,
                                                P, P, P, P, P, ctypes.POINTER(VerifyDebug), P, SZ, P]),
        "sam_spec_step": (ctypes.c_int, [P, P, I32, P, I32, P, P, I32, I32, F, U64, U64,
                                         P, P, P, P, P, ctypes.POINTER(VerifyDebug),
                                         I32, P, P, P, P, P, SZ, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = load()
    return _lib


def check(rc: int, what: str) -> None:
    if rc != OK:
        msg = lib().samspec_strerror(rc).decode()
        raise SamspecError(f"{what} failed: {rc} ({msg})")
