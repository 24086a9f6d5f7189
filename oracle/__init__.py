"""CPU oracle for the SAM-drafting + lossless-verification path.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference arm of ``bench.py`` are the only code allowed to import
this package.  The product library never loads it, and it shares no code with
the CUDA path.  The arithmetic lives in ``oracle.cpp`` (plain single-threaded
C++, fp64); this module only compiles it with the host C++ compiler and
marshals numpy arrays through ctypes.

Function map (each function cites the page passage it follows in oracle.cpp):
  Sam                 -- dynamic suffix automaton, extend + draft + dump
  verify(...)         -- greedy / rejection-sampling verification of a batch
  cdf_interval(...)   -- normalised CDF interval of one token of a residual
  tree_verify(...)    -- draft-tree verification (sibling-wise cumulative test)
  truncate_row(...)   -- per-request temperature / top-k / top-p distribution
  verify_sampling(...) -- verification against those truncated distributions
  philox4x32_10 / uniforms -- the counter-based generator behind the coins
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK = 0
ETOKEN = 3
BADROW = 5
BADDRAFT = 6
BADPARAM = 8


def build(force: bool = False) -> str:
    """Compile oracle.cpp into _build/liboracle.so (g++ -O2, no vendor flags)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P, I32, I64, U64, D = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_double
        lib.osam_new.restype = P
        lib.osam_new.argtypes = [I32]
        lib.osam_free.argtypes = [P]
        lib.osam_extend.restype = I32
        lib.osam_extend.argtypes = [P, P, I64]
        lib.osam_draft.argtypes = [P, I32, P, P]
        lib.osam_sizes.argtypes = [P, P]
        lib.osam_dump.argtypes = [P, P, P, P, P]
        lib.osam_step_batch.argtypes = [P, I32, P, P, I32, I32, P, P]
        lib.osam_match.argtypes = [P, P, P, I64, I32, P, P]
        lib.osam_match_batch.argtypes = [P, I32, P, P, P, I32, I32, P, P]
        lib.oselect_static.restype = I32
        lib.oselect_static.argtypes = [I32, I32, I32]
        lib.ophilox4x32_10.argtypes = [P, P, P]
        lib.ouniforms.argtypes = [U64, U64, I64, I32, P]
        lib.over_verify.restype = I32
        lib.over_verify.argtypes = [P, P, P, P, P, I32, I32, I32, D, U64, U64,
                                    P, P, P, P, P, P, P, P, P, P, P]
        lib.over_cdf_interval.argtypes = [P, P, I32, D, I32, I32, P]
        lib.over_tree_node_info.argtypes = [P, I32, D, P, I32, I32, P, P]
        lib.over_tree_verify.restype = I32
        lib.over_tree_verify.argtypes = [P, P, P, P, I32, I32, I32, D, U64, U64, P, P, P, P, P, P]
        lib.over_verify_sampling.restype = I32
        lib.over_verify_sampling.argtypes = [P, P, P, I32, I32, I32, P, P, P, U64, U64,
                                             P, P, P, P, P, P, P, P]
        lib.over_truncate_row.restype = I32
        lib.over_truncate_row.argtypes = [P, I32, D, I32, D, P, P]
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class Sam:
    """One dynamic suffix automaton (states numbered in creation order, the
    new state before its clone)."""

    def __init__(self, vocab: int):
        self._lib = _load()
        self._h = self._lib.osam_new(int(vocab))

    def __del__(self):
        h, self._h = getattr(self, "_h", None), None
        if h:
            self._lib.osam_free(h)

    @property
    def handle(self):
        return self._h

    def extend(self, tokens) -> int:
        t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32).reshape(-1))
        return int(self._lib.osam_extend(self._h, _ptr(t), t.size))

    def draft(self, K: int):
        out = np.empty(max(K, 1), np.int32)
        info = np.empty(3, np.int32)
        self._lib.osam_draft(self._h, int(K), _ptr(out), _ptr(info))
        return out[:K].copy(), int(info[0]), int(info[1]), int(info[2])

    def match(self, state, tokens, K: int):
        """Static use: moves the matching state (v, l) of a generated text by
        `tokens` and drafts K corpus tokens from the final state.  Returns
        ((v, l), draft [K] (-1 padded), draft_len, min_endpos)."""
        st = np.asarray(state, np.int32).copy()
        tok = np.ascontiguousarray(tokens, dtype=np.int32)
        out = np.empty(max(K, 1), np.int32)
        info = np.empty(3, np.int32)
        self._lib.osam_match(self._h, _ptr(st), _ptr(tok), tok.size, int(K), _ptr(out), _ptr(info))
        return (int(st[0]), int(st[1])), out[:K].copy(), int(info[0]), int(info[2])

    def sizes(self):
        s = np.empty(5, np.int64)
        self._lib.osam_sizes(self._h, _ptr(s))
        return dict(n_states=int(s[0]), n_edges=int(s[1]), n_tokens=int(s[2]),
                    walk_steps=int(s[3]), last=int(s[4]))

    def dump(self):
        sz = self.sizes()
        ns, ne = sz["n_states"], sz["n_edges"]
        ln = np.empty(ns, np.int32)
        lk = np.empty(ns, np.int32)
        me = np.empty(ns, np.int32)
        ed = np.empty((max(ne, 1), 3), np.int32)
        self._lib.osam_dump(self._h, _ptr(ln), _ptr(lk), _ptr(me), _ptr(ed))
        return dict(len=ln, link=lk, min_endpos=me, edges=ed[:ne].copy())


def step_batch(sams, tokens, n_new, K):
    """Extend every automaton by n_new[b] tokens of tokens[b] and draft K
    (one C call for the whole batch; used for CPU timing)."""
    lib = _load()
    B = len(sams)
    handles = (ctypes.c_void_p * B)(*[s.handle for s in sams])
    tok = np.ascontiguousarray(tokens, dtype=np.int32)
    nn = np.ascontiguousarray(n_new, dtype=np.int32)
    draft = np.empty((B, max(K, 1)), np.int32)
    info = np.empty((B, 3), np.int32)
    lib.osam_step_batch(handles, B, _ptr(tok), _ptr(nn), tok.shape[1], int(K),
                        _ptr(draft), _ptr(info))
    return draft[:, :K], info


def philox4x32_10(ctr, key):
    lib = _load()
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.empty(4, np.uint32)
    lib.ophilox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def uniforms(seed: int, step: int, b: int, j: int):
    """(u_acc, u_res) of sequence b at draft position j."""
    lib = _load()
    u = np.empty(2, np.float64)
    lib.ouniforms(int(seed), int(step), int(b), int(j), _ptr(u))
    return float(u[0]), float(u[1])


def verify(target, draft, draft_len=None, temperature=0.0, seed=0, step=0,
           draft_logits=None, seq_index=None):
    """Verify a batch.  target [B, K+1, V] (any float dtype, widened to fp32
    exactly), draft [B, K] int, optional draft_len [B], draft_logits [B, K, V].
    Returns a dict of numpy arrays (accept_len, out_token, status and the
    per-row debug values)."""
    lib = _load()
    t = np.ascontiguousarray(target, dtype=np.float32)
    B, K1, V = t.shape
    K = K1 - 1
    d = np.ascontiguousarray(np.asarray(draft, dtype=np.int32).reshape(B, K))
    dl = None if draft_len is None else np.ascontiguousarray(draft_len, dtype=np.int32)
    g = None if draft_logits is None else np.ascontiguousarray(draft_logits, dtype=np.float32)
    if g is not None:
        assert g.shape == (B, K, V)
    si = None if seq_index is None else np.ascontiguousarray(seq_index, dtype=np.int64)
    out = {k: np.empty(B, np.int32) for k in ("accept_len", "out_token", "status")}
    for k in ("row_m", "row_z", "p_d", "q_d", "u_acc"):
        out[k] = np.empty((B, K1), np.float64)
    out["row_arg"] = np.empty((B, K1), np.int32)
    out["u_res"] = np.empty(B, np.float64)
    out["res_mass"] = np.empty(B, np.float64)
    lib.over_verify(_ptr(t), _ptr(g), _ptr(d), _ptr(dl), _ptr(si), B, K, V,
                    float(temperature), int(seed) & (2**64 - 1), int(step) & (2**64 - 1),
                    _ptr(out["accept_len"]), _ptr(out["out_token"]), _ptr(out["status"]),
                    _ptr(out["row_m"]), _ptr(out["row_z"]), _ptr(out["p_d"]), _ptr(out["q_d"]),
                    _ptr(out["u_acc"]), _ptr(out["u_res"]), _ptr(out["res_mass"]),
                    _ptr(out["row_arg"]))
    return out


def cdf_interval(target_row, temperature, rejected_token, token, draft_row=None):
    """Normalised [lo, hi) CDF interval of `token` under the residual of one
    row; rejected_token < 0 means the bonus residual (r = p)."""
    lib = _load()
    t = np.ascontiguousarray(target_row, dtype=np.float32).reshape(-1)
    g = None if draft_row is None else np.ascontiguousarray(draft_row, dtype=np.float32).reshape(-1)
    res = np.empty(3, np.float64)
    lib.over_cdf_interval(_ptr(t), _ptr(g), t.size, float(temperature), int(rejected_token),
                          int(token), _ptr(res))
    return float(res[0]), float(res[1]), float(res[2])


def match_batch(sam, state, tokens, n_new, K):
    """sam.match for B texts in one C call (timing): state int32 [B, 2] is
    updated in place; returns draft [B, K] and info [B, 3] (draft_len, match
    length, min_endpos)."""
    lib = _load()
    tok = np.ascontiguousarray(tokens, dtype=np.int32)
    nn = np.ascontiguousarray(n_new, dtype=np.int32)
    B = len(nn)
    draft = np.empty((B, max(K, 1)), np.int32)
    info = np.empty((B, 3), np.int32)
    lib.osam_match_batch(sam._h, B, _ptr(state), _ptr(tok), _ptr(nn), tok.shape[1], int(K),
                         _ptr(draft), _ptr(info))
    return draft[:, :K], info


def select_static(l_static: int, l_dynamic: int, l_bias: int) -> bool:
    """Adaptive choice between a static and a dynamic automaton's drafts: the
    static draft only when its match is longer by more than l_bias."""
    return bool(_load().oselect_static(int(l_static), int(l_dynamic), int(l_bias)))


def tree_verify(target, tok, first_child, next_sibling, temperature=0.0, seed=0, step=0):
    """Verify a draft tree per sequence.  target [B, N, V] (row n: the token
    after node n's path), tok / first_child / next_sibling [B, N] int (node 0
    the verified context; -1 links: none).  Returns accept_len, out_token,
    path [B, N] (accepted node indices, -1 after), status, u_res, res_mass."""
    lib = _load()
    t = np.ascontiguousarray(target, dtype=np.float32)
    B, N, V = t.shape
    tk = np.ascontiguousarray(tok, dtype=np.int32).reshape(B, N)
    fc = np.ascontiguousarray(first_child, dtype=np.int32).reshape(B, N)
    ns = np.ascontiguousarray(next_sibling, dtype=np.int32).reshape(B, N)
    out = {k: np.empty(B, np.int32) for k in ("accept_len", "out_token", "status")}
    out["path"] = np.empty((B, N), np.int32)
    out["u_res"] = np.empty(B, np.float64)
    out["res_mass"] = np.empty(B, np.float64)
    lib.over_tree_verify(_ptr(t), _ptr(tk), _ptr(fc), _ptr(ns), B, N, V, float(temperature),
                         int(seed) & (2**64 - 1), int(step) & (2**64 - 1), _ptr(out["accept_len"]),
                         _ptr(out["out_token"]), _ptr(out["path"]), _ptr(out["status"]),
                         _ptr(out["u_res"]), _ptr(out["res_mass"]))
    return out


def tree_node_info(row, temperature, children, token):
    """At one tree node: cumulative probabilities of its children (sibling
    order) and the [lo, hi) interval of `token` in the node's final-sample
    distribution (children removed).  Returns (acc [n], lo, hi, mass)."""
    lib = _load()
    r = np.ascontiguousarray(row, dtype=np.float32)
    ch = np.ascontiguousarray(children, dtype=np.int32)
    acc = np.empty(max(len(ch), 1), np.float64)
    lhm = np.empty(3, np.float64)
    lib.over_tree_node_info(_ptr(r), r.size, float(temperature), _ptr(ch), len(ch), int(token),
                            _ptr(acc), _ptr(lhm))
    return acc[:len(ch)], float(lhm[0]), float(lhm[1]), float(lhm[2])


def truncate_row(row, temperature, top_k=0, top_p=1.0):
    """One row's distribution under per-request sampling parameters:
    softmax(l / T), top-k renormalisation, top-p renormalisation.  Returns
    (p' [V] float64, tau) with tau the smallest kept logit; None for a bad
    row."""
    lib = _load()
    r = np.ascontiguousarray(row, dtype=np.float32).reshape(-1)
    pp = np.empty(r.size, np.float64)
    tau = np.empty(1, np.float32)
    rc = lib.over_truncate_row(_ptr(r), r.size, float(temperature), int(top_k), float(top_p),
                               _ptr(pp), _ptr(tau))
    return None if rc != 0 else (pp, float(tau[0]))


def verify_sampling(target, draft, draft_len=None, temperature=None, top_k=None, top_p=None,
                    seed=0, step=0):
    """Verify one-hot drafts against per-request truncated distributions.
    target [B, K+1, V]; draft [B, K]; temperature, top_k, top_p: [B] (top_k
    <= 0 or >= V and top_p >= 1 disable truncation).  Returns accept_len,
    out_token, status, p_d / u_acc / tau [B, K+1], u_res, res_mass."""
    lib = _load()
    t = np.ascontiguousarray(target, dtype=np.float32)
    B, K1, V = t.shape
    K = K1 - 1
    d = np.ascontiguousarray(np.asarray(draft, dtype=np.int32).reshape(B, K))
    dl = None if draft_len is None else np.ascontiguousarray(draft_len, dtype=np.int32)
    T = np.ascontiguousarray(np.broadcast_to(1.0 if temperature is None else temperature, (B,)),
                             dtype=np.float64)
    tk = np.ascontiguousarray(np.broadcast_to(0 if top_k is None else top_k, (B,)), dtype=np.int32)
    tp = np.ascontiguousarray(np.broadcast_to(1.0 if top_p is None else top_p, (B,)), dtype=np.float64)
    out = {k: np.empty(B, np.int32) for k in ("accept_len", "out_token", "status")}
    for k in ("p_d", "u_acc"):
        out[k] = np.empty((B, K1), np.float64)
    out["tau"] = np.empty((B, K1), np.float32)
    out["u_res"] = np.empty(B, np.float64)
    out["res_mass"] = np.empty(B, np.float64)
    lib.over_verify_sampling(_ptr(t), _ptr(d), _ptr(dl), B, K, V, _ptr(T), _ptr(tk), _ptr(tp),
                             int(seed) & (2**64 - 1), int(step) & (2**64 - 1),
                             _ptr(out["accept_len"]), _ptr(out["out_token"]), _ptr(out["status"]),
                             _ptr(out["p_d"]), _ptr(out["u_acc"]), _ptr(out["u_res"]),
                             _ptr(out["res_mass"]), _ptr(out["tau"]))
    return out
