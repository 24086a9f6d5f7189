"""GB300-native SAM drafting and lossless speculative verification.

Python face of libsamspec.so (C ABI in include/samspec.h).  The same names as
the C entry points, over torch CUDA tensors:

  SamBatch(B, capacity_tokens, vocab)   -- sam_batch_create / _destroy
    .extend(tokens, n_new)              -- sam_extend
    .draft(K)                           -- sam_draft
    .step(tokens, n_new, K)             -- sam_step (extend + draft, one launch)
    .step_rows(rows, tokens, n_new, K)  -- sam_step_rows (a subset of the sequences)
    .spec_step(target, draft, ...)      -- sam_spec_step (verify, extend, draft)
    .match(row, state, tokens, n_new, K) -- ssam_match (a corpus automaton, static use)
  select_drafts(dynamic, static, l_bias) -- sam_select_drafts
    .status(), .reset(mask), .dump(b), .export(), .import_(blob)
  spec_verify(target, draft, ...)       -- spec_verify
  spec_verify_tree(target, tok, ...)    -- spec_verify_tree (draft trees)
  spec_uniforms(B, K, seed, step)       -- spec_uniforms

Device memory (workspaces, inputs, outputs) comes from torch; each call is
enqueued on torch's current CUDA stream.
"""
from __future__ import annotations

import ctypes

import torch

from . import _binding as _b
from ._binding import (BF16, F32, ST_BADDRAFT, ST_BADROW, ST_CAPACITY, ST_HASHFULL,  # noqa: F401
                       ST_LOOPCAP, ST_OK, ST_TIMEOUT, ST_TOKEN, SamspecError)

__all__ = ["SamBatch", "spec_verify", "spec_verify_tree", "spec_uniforms", "select_drafts",
           "SamspecError", "library_path"]


def library_path() -> str:
    return _b.LIB_PATH


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device=None):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _is_cuda(t):
    return t.is_cuda


def _req(t, dtype, name, shape=None, device=None):
    """t, checked: a contiguous CUDA tensor of `dtype` (and `shape`, on
    `device`, where given) -- the kernels take its pointer as it is."""
    if not isinstance(t, torch.Tensor) or not _is_cuda(t):
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    return t


def _need(res, key, shape, dev, dtype=torch.int32, fill=None):
    """res[key]: the caller's output buffer, checked, or a new one."""
    if key in res:
        _req(res[key], dtype, f"out[{key}]", shape, dev)
    else:
        res[key] = (torch.empty(shape, dtype=dtype, device=dev) if fill is None
                    else torch.full(shape, fill, dtype=dtype, device=dev))


def _cuda_device(device=None):
    """torch.device of a CUDA device, with its index."""
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    if dev.type == "cuda" and dev.index is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    return dev


def _workspace(workspace, B, K, V, dev, sampling=False):
    """The caller's verification workspace, checked, or the cached one."""
    if workspace is None:
        return verify_workspace(B, K, V, dev, sampling=sampling)
    return _req(workspace, torch.uint8, "workspace", None, dev)


class SamBatch:
    """B device-resident dynamic suffix automata (one per sequence)."""

    def __init__(self, B: int, capacity_tokens: int, vocab: int, device=None):
        self.lib = _b.lib()
        self.B, self.C, self.V = int(B), int(capacity_tokens), int(vocab)
        self.device = _cuda_device(device)
        nbytes = self.lib.sam_batch_workspace_bytes(self.B, self.C)
        if nbytes == 0:
            raise SamspecError(f"sizes outside the limits: B={B}, capacity={capacity_tokens}")
        self.ws_bytes = int(nbytes)
        self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, device=self.device)
        h = ctypes.c_void_p()
        with torch.cuda.device(self.device):
            _b.check(self.lib.sam_batch_create(self.B, self.C, self.V, _ptr(self.workspace),
                                               self.ws_bytes, _stream(self.device), ctypes.byref(h)),
                     "sam_batch_create")
        self._h = h

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            self.lib.sam_batch_destroy(h)
            self._h = None

    def reset(self, mask=None):
        if mask is not None:
            _req(mask, torch.int32, "mask", (self.B,), self.device)
        _b.check(self.lib.sam_reset(self._h, _ptr(mask), _stream(self.device)), "sam_reset")

    def extend(self, tokens, n_new):
        _req(tokens, torch.int32, "tokens", device=self.device)
        if tokens.dim() != 2 or tokens.shape[0] != self.B:
            raise ValueError("tokens must be [B, max_new]")
        _req(n_new, torch.int32, "n_new", (self.B,), self.device)
        _b.check(self.lib.sam_extend(self._h, _ptr(tokens), _ptr(n_new), int(tokens.shape[1]),
                                     _stream(self.device)), "sam_extend")

    def _outs(self, K, out):
        if out is None:
            z = lambda *s: torch.empty(s, dtype=torch.int32, device=self.device)  # noqa: E731
            out = (z(self.B, K), z(self.B), z(self.B), z(self.B))
        d, dl, ml, me = out
        _req(d, torch.int32, "draft", (self.B, K), self.device)
        for t, n in ((dl, "draft_len"), (ml, "match_len"), (me, "min_endpos")):
            if t is not None:
                _req(t, torch.int32, n, (self.B,), self.device)
        return out

    def _outs_n(self, n, K, out):
        """Output buffers of n sequences: the caller's, checked, or new ones."""
        if out is None:
            z = lambda *s: torch.empty(s, dtype=torch.int32, device=self.device)  # noqa: E731
            return z(n, K), z(n), z(n), z(n)
        d, dl, ml, me = out
        _req(d, torch.int32, "draft", (n, K), self.device)
        for t, nm in ((dl, "draft_len"), (ml, "match_len"), (me, "min_endpos")):
            if t is not None:
                _req(t, torch.int32, nm, (n,), self.device)
        return out

    def draft(self, K: int, out=None):
        d, dl, ml, me = self._outs(K, out)
        _b.check(self.lib.sam_draft(self._h, int(K), _ptr(d), _ptr(dl), _ptr(ml), _ptr(me),
                                    _stream(self.device)), "sam_draft")
        return d, dl, ml, me

    def step(self, tokens, n_new, K: int, out=None):
        _req(tokens, torch.int32, "tokens", device=self.device)
        if tokens.dim() != 2 or tokens.shape[0] != self.B:
            raise ValueError("tokens must be [B, max_new]")
        _req(n_new, torch.int32, "n_new", (self.B,), self.device)
        d, dl, ml, me = self._outs(K, out)
        _b.check(self.lib.sam_step(self._h, _ptr(tokens), _ptr(n_new), int(tokens.shape[1]), int(K),
                                   _ptr(d), _ptr(dl), _ptr(ml), _ptr(me), _stream(self.device)),
                 "sam_step")
        return d, dl, ml, me

    def step_rows(self, rows, tokens, n_new, K: int, out=None):
        """sam_step on the automata `rows` (int32 [n], or None for 0..n-1)."""
        _req(tokens, torch.int32, "tokens", device=self.device)
        if tokens.dim() != 2:
            raise ValueError("tokens must be [n, max_new]")
        n = int(tokens.shape[0])
        if rows is not None:
            _req(rows, torch.int32, "rows", (n,), self.device)
        _req(n_new, torch.int32, "n_new", (n,), self.device)
        d, dl, ml, me = self._outs_n(n, K, out)
        _b.check(self.lib.sam_step_rows(self._h, _ptr(rows), n, _ptr(tokens), _ptr(n_new),
                                        int(tokens.shape[1]), int(K), _ptr(d) if K > 0 else None,
                                        _ptr(dl), _ptr(ml), _ptr(me), _stream(self.device)),
                 "sam_step_rows")
        return d, dl, ml, me

    def spec_step(self, target, draft, draft_len=None, K_next: int = 3, rows=None,
                  temperature: float = 0.0, seed: int = 0, step: int = 0, out=None,
                  workspace=None):
        """One decode step: verify `draft` ([n, K], one-hot) against `target`
        ([n, K+1, V]), extend each automaton by its emitted tokens, draft
        K_next tokens.  Returns a dict of CUDA tensors (accept_len, out_token,
        emit, emit_len, status, next_draft, next_draft_len, match_len,
        min_endpos)."""
        if target.dim() != 3:
            raise ValueError("target must be [n, K+1, V]")
        n, K1, V = (int(x) for x in target.shape)
        K = K1 - 1
        dt = {torch.float32: F32, torch.bfloat16: BF16}.get(target.dtype)
        if dt is None:
            raise TypeError("target must be float32 or bfloat16")
        dev = self.device
        _req(target, target.dtype, "target", device=dev)
        _req(draft, torch.int32, "draft", (n, K), dev)
        if draft_len is not None:
            _req(draft_len, torch.int32, "draft_len", (n,), dev)
        if rows is not None:
            _req(rows, torch.int32, "rows", (n,), dev)
        res = out if out is not None else {}
        for k in ("accept_len", "out_token", "emit_len", "status", "next_draft_len", "match_len",
                  "min_endpos"):
            _need(res, k, (n,), dev)
        _need(res, "emit", (n, K1), dev)
        _need(res, "next_draft", (n, int(K_next)), dev)
        ws = _workspace(workspace, n, K, V, dev)
        _b.check(self.lib.sam_spec_step(
            self._h, _ptr(rows), n, _ptr(target), dt, _ptr(draft) if K > 0 else None,
            _ptr(draft_len), K, V, float(temperature), int(seed) & (2**64 - 1),
            int(step) & (2**64 - 1), _ptr(res["accept_len"]), _ptr(res["out_token"]),
            _ptr(res["emit"]), _ptr(res["emit_len"]), _ptr(res["status"]), None, int(K_next),
            _ptr(res["next_draft"]) if K_next > 0 else None, _ptr(res["next_draft_len"]),
            _ptr(res["match_len"]), _ptr(res["min_endpos"]), _ptr(ws), ws.numel(),
            _stream(self.device)), "sam_spec_step")
        return res

    def match(self, row: int, state, tokens, n_new, K: int, out=None):
        """Static use of automaton `row` (a corpus): moves the matching states
        `state` (int32 [n, 2], in place) by tokens [n, max_new] / n_new [n] and
        drafts K corpus tokens.  Returns (draft, draft_len, match_len,
        min_endpos)."""
        _req(state, torch.int32, "state", device=self.device)
        if state.dim() != 2 or state.shape[1] != 2:
            raise ValueError("state must be [n, 2]")
        n = int(state.shape[0])
        _req(tokens, torch.int32, "tokens", device=self.device)
        if tokens.dim() != 2 or tokens.shape[0] != n:
            raise ValueError("tokens must be [n, max_new]")
        _req(n_new, torch.int32, "n_new", (n,), self.device)
        d, dl, ml, me = self._outs_n(n, K, out)
        _b.check(self.lib.ssam_match(self._h, int(row), n, _ptr(state), _ptr(tokens), _ptr(n_new),
                                     int(tokens.shape[1]), int(K), _ptr(d) if K > 0 else None,
                                     _ptr(dl), _ptr(ml), _ptr(me), _stream(self.device)),
                 "ssam_match")
        return d, dl, ml, me

    def status(self):
        import numpy as np
        out = np.empty(self.B, np.int32)
        _b.check(self.lib.sam_get_status(self._h, out.ctypes.data_as(ctypes.c_void_p),
                                         _stream(self.device)), "sam_get_status")
        return out

    def export(self):
        blob = torch.empty(self.ws_bytes, dtype=torch.uint8, device=self.device)
        _b.check(self.lib.sam_export(self._h, _ptr(blob), self.ws_bytes, _stream(self.device)),
                 "sam_export")
        return blob

    def import_(self, blob):
        _req(blob, torch.uint8, "blob", device=self.device)
        _b.check(self.lib.sam_import(self._h, _ptr(blob), blob.numel(), _stream(self.device)),
                 "sam_import")

    def dump(self, b: int):
        """Sequence b's automaton as numpy arrays (synchronises)."""
        import numpy as np
        sc = np.zeros(8, np.int32)
        _b.check(self.lib.sam_dump_sequence(self._h, int(b), sc.ctypes.data_as(ctypes.c_void_p),
                                            None, None, None, 0, None, 0, _stream(self.device)),
                 "sam_dump_sequence")
        ns, ne = int(sc[2]), int(sc[3])
        ln = np.empty(max(ns, 1), np.int32)
        lk = np.empty(max(ns, 1), np.int32)
        me = np.empty(max(ns, 1), np.int32)
        ed = np.empty((max(ne, 1), 3), np.int32)
        vp = lambda a: a.ctypes.data_as(ctypes.c_void_p)  # noqa: E731
        _b.check(self.lib.sam_dump_sequence(self._h, int(b), vp(sc), vp(ln), vp(lk), vp(me), ns,
                                            vp(ed), ne, _stream(self.device)), "sam_dump_sequence")
        return dict(n_tokens=int(sc[0]), last=int(sc[1]), n_states=ns, n_edges=ne,
                    status=int(sc[4]), len=ln[:ns], link=lk[:ns], min_endpos=me[:ns],
                    edges=ed[:ne])


_ws_cache = {}
# workspaces replaced in the cache by a larger one: kept allocated, since a
# CUDA graph captured with the smaller one may still be replayed
_ws_retired = []


def verify_workspace(B: int, K: int, V: int, device=None, sampling: bool = False):
    """A zero-initialised verification workspace, cached per (device, stream);
    sampling=True sizes it for spec_verify_sampling.  A cached workspace is
    never freed (a larger need replaces it in the cache only), so graphs
    captured with it stay valid; a workspace the caller allocates must stay
    allocated while any graph that uses it can still be replayed."""
    lib = _b.lib()
    dev = _cuda_device(device)
    need = int(lib.spec_verify_sampling_workspace_bytes(B, K, V) if sampling
               else lib.spec_verify_workspace_bytes(B, K, V))
    key = (dev.index, torch.cuda.current_stream(dev).cuda_stream)
    ws = _ws_cache.get(key)
    if ws is None or ws.numel() < need:
        if ws is not None:
            _ws_retired.append(ws)
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
        _b.check(lib.spec_verify_workspace_init(_ptr(ws), ws.numel(), _stream(dev)),
                 "spec_verify_workspace_init")
        _ws_cache[key] = ws
    return ws


def spec_verify(target, draft, draft_len=None, temperature: float = 0.0, seed: int = 0,
                step: int = 0, draft_logits=None, out=None, emit: bool = False,
                status: bool = True, debug: bool = False, workspace=None):
    """Verify K drafts per sequence against target logits [B, K+1, V].

    Returns a dict of CUDA tensors: accept_len, out_token (+ emit, emit_len,
    status, and the debug rows row_m, row_z, p_d, q_d, row_arg, res_mass)."""
    lib = _b.lib()
    if target.dim() != 3:
        raise ValueError("target must be [B, K+1, V]")
    B, K1, V = (int(x) for x in target.shape)
    K = K1 - 1
    dt = {torch.float32: F32, torch.bfloat16: BF16}.get(target.dtype)
    if dt is None:
        raise TypeError("target must be float32 or bfloat16")
    _req(target, target.dtype, "target")
    dev = target.device
    _req(draft, torch.int32, "draft", (B, K), dev)
    if draft_len is not None:
        _req(draft_len, torch.int32, "draft_len", (B,), dev)
    ddt = F32
    if draft_logits is not None:
        ddt = {torch.float32: F32, torch.bfloat16: BF16}.get(draft_logits.dtype)
        if ddt is None:
            raise TypeError("draft_logits must be float32 or bfloat16")
        _req(draft_logits, draft_logits.dtype, "draft_logits", (B, K, V), dev)
    res = out if out is not None else {}
    # the caller's buffers are checked and reused; the others are allocated
    _need(res, "accept_len", (B,), dev)
    _need(res, "out_token", (B,), dev)
    for key, shape in (("emit", (B, K1)), ("emit_len", (B,))):
        if emit or key in res:
            _need(res, key, shape, dev)
    if status or "status" in res:
        _need(res, "status", (B,), dev)
    dbg = None
    if debug:
        for k in ("row_m", "row_z", "p_d", "q_d"):
            _need(res, k, (B, K1), dev, torch.float32, float("nan"))
        _need(res, "row_arg", (B, K1), dev, torch.int32, -1)
        _need(res, "res_mass", (B,), dev, torch.float32, float("nan"))
        dbg = _b.VerifyDebug(*[res[k].data_ptr() for k in ("row_m", "row_z", "p_d", "q_d", "row_arg", "res_mass")])
    ws = _workspace(workspace, B, K, V, dev)
    rc = lib.spec_verify(_ptr(target), dt, _ptr(draft_logits), ddt, _ptr(draft) if K > 0 else None,
                         _ptr(draft_len),
                         B, K, V, float(temperature), int(seed) & (2**64 - 1), int(step) & (2**64 - 1),
                         _ptr(res["accept_len"]), _ptr(res["out_token"]), _ptr(res.get("emit")),
                         _ptr(res.get("emit_len")), _ptr(res.get("status")),
                         ctypes.byref(dbg) if dbg is not None else None,
                         _ptr(ws), ws.numel(), _stream(dev))
    _b.check(rc, "spec_verify")
    return res


def select_drafts(dynamic, static, l_bias: int):
    """Per sequence, the static automaton's draft when its match is longer than
    the dynamic one's by more than l_bias, else the dynamic draft.  dynamic /
    static: (draft [n, K], draft_len [n], match_len [n]).  Returns (draft,
    draft_len, source) with source 1 where the static draft was taken."""
    dd, dl, dm = dynamic
    sd, sl, sm = static
    _req(dd, torch.int32, "dynamic draft")
    if dd.dim() != 2:
        raise ValueError("dynamic draft must be [n, K]")
    n, K = (int(x) for x in dd.shape)
    dev = dd.device
    _req(sd, torch.int32, "static draft", (n, K), dev)
    for t, nm in ((dl, "dynamic draft_len"), (dm, "dynamic match_len"), (sl, "static draft_len"),
                  (sm, "static match_len")):
        _req(t, torch.int32, nm, (n,), dev)
    od = torch.empty_like(dd)
    ol = torch.empty_like(dl)
    src = torch.empty_like(dl)
    _b.check(_b.lib().sam_select_drafts(n, K, _ptr(dd), _ptr(dl), _ptr(dm), _ptr(sd), _ptr(sl),
                                        _ptr(sm), int(l_bias), _ptr(od), _ptr(ol), _ptr(src),
                                        _stream(dd.device)), "sam_select_drafts")
    return od, ol, src


def spec_verify_tree(target, tok, first_child, next_sibling, temperature: float = 0.0,
                     seed: int = 0, step: int = 0, debug: bool = False, workspace=None, out=None):
    """Verify a draft tree per sequence: target [B, N, V] (row n: the token
    after node n's path), tok / first_child / next_sibling int32 [B, N].
    Returns a dict of CUDA tensors: accept_len, out_token, path [B, N], emit
    [B, N], emit_len, status (+ row_m, row_z, row_arg, res_mass).  `out`: the
    dict of an earlier call with the same sizes, written again in place."""
    lib = _b.lib()
    if target.dim() != 3:
        raise ValueError("target must be [B, N, V]")
    B, N, V = (int(x) for x in target.shape)
    dt = {torch.float32: F32, torch.bfloat16: BF16}.get(target.dtype)
    if dt is None:
        raise TypeError("target must be float32 or bfloat16")
    _req(target, target.dtype, "target")
    dev = target.device
    for t, nm in ((tok, "tok"), (first_child, "first_child"), (next_sibling, "next_sibling")):
        _req(t, torch.int32, nm, (B, N), dev)
    res = out if out is not None else {}
    for k, shp in (("accept_len", (B,)), ("out_token", (B,)), ("path", (B, N)), ("emit", (B, N)),
                   ("emit_len", (B,)), ("status", (B,))):
        _need(res, k, shp, dev)
    dbg = None
    if debug:
        for k in ("row_m", "row_z"):
            res[k] = torch.full((B, N), float("nan"), dtype=torch.float32, device=dev)
        res["row_arg"] = torch.full((B, N), -1, dtype=torch.int32, device=dev)
        res["res_mass"] = torch.full((B,), float("nan"), dtype=torch.float32, device=dev)
        dbg = _b.VerifyDebug(res["row_m"].data_ptr(), res["row_z"].data_ptr(), 0, 0,
                             res["row_arg"].data_ptr(), res["res_mass"].data_ptr())
    ws = _workspace(workspace, B, N - 1, V, dev)
    _b.check(lib.spec_verify_tree(_ptr(target), dt, _ptr(tok), _ptr(first_child), _ptr(next_sibling),
                                  B, N, V, float(temperature), int(seed) & (2**64 - 1),
                                  int(step) & (2**64 - 1), _ptr(res["accept_len"]), _ptr(res["out_token"]),
                                  _ptr(res["path"]), _ptr(res["emit"]), _ptr(res["emit_len"]),
                                  _ptr(res["status"]), ctypes.byref(dbg) if dbg is not None else None,
                                  _ptr(ws), ws.numel(), _stream(dev)), "spec_verify_tree")
    return res


def _per_seq(x, B, dtype, dev, name):
    """A [B] device tensor of `dtype` from a scalar or a [B] tensor."""
    if isinstance(x, torch.Tensor):
        return _req(x, dtype, name, (B,), dev)
    return torch.full((B,), x, dtype=dtype, device=dev)


def sampling_cut(target, temperature, top_k, top_p):
    """The cut of each row [B, R, V] under per-sequence (temperature, top_k,
    top_p) ([B] tensors or scalars): [B, R] float32 tau, the smallest kept
    logit (-inf: nothing cut; NaN: bad parameters)."""
    lib = _b.lib()
    if target.dim() != 3:
        raise ValueError("target must be [B, R, V]")
    B, R, V = (int(x) for x in target.shape)
    dt = {torch.float32: F32, torch.bfloat16: BF16}.get(target.dtype)
    if dt is None:
        raise TypeError("target must be float32 or bfloat16")
    _req(target, target.dtype, "target")
    dev = target.device
    T = _per_seq(temperature, B, torch.float32, dev, "temperature")
    k = _per_seq(top_k, B, torch.int32, dev, "top_k")
    p = _per_seq(top_p, B, torch.float32, dev, "top_p")
    tau = torch.empty((B, R), dtype=torch.float32, device=dev)
    _b.check(lib.spec_sampling_cut(_ptr(target), dt, B, R, V, _ptr(T), _ptr(k), _ptr(p), _ptr(tau),
                                   _stream(dev)), "spec_sampling_cut")
    return tau


def spec_verify_sampling(target, draft, draft_len=None, temperature=1.0, top_k=0, top_p=1.0,
                         seed: int = 0, step: int = 0, out=None, emit: bool = False,
                         debug: bool = False, workspace=None):
    """Verify one-hot drafts [B, K] against target logits [B, K+1, V] with
    per-sequence temperature, top_k and top_p ([B] tensors or scalars).
    Returns a dict of CUDA tensors: accept_len, out_token, status (+ emit,
    emit_len, and the debug rows row_m, row_z, p_d, row_arg, res_mass)."""
    lib = _b.lib()
    if target.dim() != 3:
        raise ValueError("target must be [B, K+1, V]")
    B, K1, V = (int(x) for x in target.shape)
    K = K1 - 1
    dt = {torch.float32: F32, torch.bfloat16: BF16}.get(target.dtype)
    if dt is None:
        raise TypeError("target must be float32 or bfloat16")
    _req(target, target.dtype, "target")
    dev = target.device
    _req(draft, torch.int32, "draft", (B, K), dev)
    if draft_len is not None:
        _req(draft_len, torch.int32, "draft_len", (B,), dev)
    T = _per_seq(temperature, B, torch.float32, dev, "temperature")
    k = _per_seq(top_k, B, torch.int32, dev, "top_k")
    p = _per_seq(top_p, B, torch.float32, dev, "top_p")
    res = out if out is not None else {}
    for key in ("accept_len", "out_token", "status"):
        _need(res, key, (B,), dev)
    for key, shape in (("emit", (B, K1)), ("emit_len", (B,))):
        if emit or key in res:
            _need(res, key, shape, dev)
    dbg = None
    if debug:
        for key in ("row_m", "row_z", "p_d"):
            _need(res, key, (B, K1), dev, torch.float32, float("nan"))
        _need(res, "row_arg", (B, K1), dev, torch.int32, -1)
        _need(res, "res_mass", (B,), dev, torch.float32, float("nan"))
        dbg = _b.VerifyDebug(res["row_m"].data_ptr(), res["row_z"].data_ptr(), res["p_d"].data_ptr(), 0,
                             res["row_arg"].data_ptr(), res["res_mass"].data_ptr())
    ws = _workspace(workspace, B, K, V, dev, sampling=True)
    rc = lib.spec_verify_sampling(_ptr(target), dt, _ptr(draft) if K > 0 else None, _ptr(draft_len),
                                  B, K, V, _ptr(T), _ptr(k), _ptr(p), int(seed) & (2**64 - 1),
                                  int(step) & (2**64 - 1), _ptr(res["accept_len"]),
                                  _ptr(res["out_token"]), _ptr(res.get("emit")),
                                  _ptr(res.get("emit_len")), _ptr(res["status"]),
                                  ctypes.byref(dbg) if dbg is not None else None,
                                  _ptr(ws), ws.numel(), _stream(dev))
    _b.check(rc, "spec_verify_sampling")
    return res


def spec_uniforms(B: int, K: int, seed: int, step: int, device=None):
    """[B, K+1, 2] float32: (u_j, u'_j) exactly as spec_verify draws them."""
    dev = _cuda_device(device)
    u = torch.empty((B, K + 1, 2), dtype=torch.float32, device=dev)
    _b.check(_b.lib().spec_uniforms(int(B), int(K), int(seed) & (2**64 - 1), int(step) & (2**64 - 1),
                                    _ptr(u), _stream(dev)), "spec_uniforms")
    return u
