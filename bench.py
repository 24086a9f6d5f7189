"""Benchmark of the SAM-drafting + lossless-verification hot path on GB300.

Default line (workload verify_b1024): lossless verification of B=1024
sequences per GPU, K=3 one-hot drafts each, V=151936, bf16 target logits
N(0, sd 2) with every draft drawn uniformly among its row's top 5, rejection
sampling at T=1.0.  One step = one spec_verify launch over the whole batch:
row statistics, the accept chain, the resample or bonus token and the Philox
coins, in one kernel.  Logits rotate through three step tensors of 1.25 GB
each (far above the 129 MB L2), and the timed region replays a CUDA graph of
exactly --steps steps, each replay bracketed by a barrier and a device
synchronisation and timed with CUDA events on the capture stream; the line
reports the median replay (max over ranks), over enough replays for at least
half a second of timed work.

The same run measures the rest of the path and puts it under `breakdown`:
  step_b64          the full decode step at B=64 (device suffix automata
                    extended by the emitted tokens and drafting K=3, then
                    verification at T=1 of bf16 logits with the continuation
                    boosted), beside the oracle on one host core and on all;
  sam_rollout_b256  the automata alone on 256 histories of 16k-32k tokens:
                    prefill tokens/s and ns per sequence-step of 512 steps of
                    extend (1-4 tokens) + draft, beside the oracle's build and
                    step on one core and on all;
  sweep_b1024       K in {1,3,5,8} x fp32/bf16 x {greedy, T=1, every row read};
  draft_model_b32   verification with draft-model logits (B=32, K=5, fp32,
                    T=0.7, residual resampling).
Under torchrun every rank runs its own batches (weak scaling, no collective on
the data path).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                  [--workload verify_b1024|rs_bf16_b64|sweep_b1024|long_rollout_b256|
                              draft_model_b32|rollout_toy_b64|static_match_b256|
                              tree_b256|sampling_b256]
"""
from __future__ import annotations

import argparse
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "verified sequence-steps/s and spec_verify HBM GB/s vs 8 TB/s; SAM ns/seq-step"
POOL = 16

# the default line's workload
HEAD_B, HEAD_K, HEAD_T = 1024, 3, 1.0
HEAD_POOL = 3
HEAD_SEED = 7303
HEAD_COIN_SEED = 5
HEAD_WORKLOAD = "verify_b1024_k3_bf16_t1"
HEAD_MIN_TIMED_MS = 500.0

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per launch of the
# verify kernel from one ncu capture of each workload, with the SHA-256 of the
# code of the translation unit it was taken on (verify.cu and every header it
# includes; comments and blank lines left out, see _code_sha256): a changed
# kernel reports null until captured again.
_VERIFY_TU = "10209560a99b9cc8583f03087bc0f389234495d313e9f20d9306041be47c2231"
VERIFY_TRAFFIC = {
    "verify_b1024_k3_bf16_t1": {"bytes": 317743872.0, "code_sha256": _VERIFY_TU},
    "draft_model_b32": {"bytes": 86080512.0, "code_sha256": _VERIFY_TU},
    "rs_bf16_b64": {"bytes": 19564800.0, "code_sha256": _VERIFY_TU},
    "long_rollout_b256": {"bytes": 78983744.0, "code_sha256": _VERIFY_TU},
    "tree_b256": {"bytes": 161326336.0, "code_sha256": _VERIFY_TU},
}
# the same for the sampling cut kernel (sampling.cu and its headers)
CUT_TRAFFIC = {"sampling_b256": {"bytes": 277508096.0,
                                 "code_sha256": "80868dc4d90963fa9ff9dc55167b6e2d48b049d28b8d7ebe5bffb0d539c8f2da"}}

CSRC = os.path.join(ROOT, "sam_drafting_verification_gb300", "csrc")
INCLUDE = os.path.join(ROOT, "include")
_INCLUDE_RE = re.compile(r'^[ \t]*#[ \t]*include[ \t]+"([^"]+)"', re.M)


def _strip_comments(text):
    """C/C++/CUDA source without its // and /* */ comments; string and
    character literals are kept as they are."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        elif c in "\"'":
            j = i + 1
            while j < n and text[j] != c and text[j] != "\n":
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(c)
            i += 1
    return "".join(out)


def _tu_sources(source):
    """A CUDA source of the library and every header it includes with quotes,
    recursively (looked up in csrc/, then include/), each once."""
    order, todo = [], [os.path.join(CSRC, source)]
    while todo:
        path = todo.pop(0)
        if path in order:
            continue
        order.append(path)
        with open(path, encoding="utf-8") as f:
            names = _INCLUDE_RE.findall(_strip_comments(f.read()))
        for name in names:
            found = [os.path.join(d, name) for d in (CSRC, INCLUDE) if os.path.exists(os.path.join(d, name))]
            if not found:
                raise FileNotFoundError(f"{name}, included by {path}")
            todo.append(found[0])
    return order


def _code_sha256(*paths):
    """SHA-256 of the code of the given sources: comments cut, trailing blanks
    cut, empty lines left out, each file's code preceded by its name, so that
    a comment edit keeps a capture valid and any code edit does not."""
    import hashlib
    h = hashlib.sha256()
    for path in paths:
        with open(path, encoding="utf-8") as f:
            lines = [ln.rstrip() for ln in _strip_comments(f.read()).split("\n")]
        h.update(os.path.basename(str(path)).encode() + b"\0")
        h.update("\n".join(ln for ln in lines if ln).encode() + b"\0")
    return h.hexdigest()


def _tu_code_sha256(source):
    return _code_sha256(*_tu_sources(source))


def _traffic(table, workload, source):
    t = table.get(workload)
    if t is None or _tu_code_sha256(source) != t["code_sha256"]:
        return None
    return t["bytes"]


def _verify_traffic(workload):
    return _traffic(VERIFY_TRAFFIC, workload, "verify.cu")


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _nproc() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None
        self.th = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.th = threading.Thread(target=self._read, daemon=True)
        self.th.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 7:
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.th.join(timeout=5)
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[3 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(self.rows)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(x, ws, device):
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _sum_over_ranks(x, ws, device):
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# --------------------------------------------------------------------------
# graphs and their timing
# --------------------------------------------------------------------------

def _capture(dev, fn, n):
    """A CUDA graph of fn(0) .. fn(n - 1), captured on a side stream."""
    import torch
    cs = torch.cuda.Stream(device=dev)
    g = torch.cuda.CUDAGraph()
    cs.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(cs):
        with torch.cuda.graph(g, stream=cs):
            for i in range(n):
                fn(i)
    torch.cuda.synchronize(dev)
    return g, cs


def _replay_ms(g, cs, ws, pre=None):
    """One replay of g on its stream, bracketed by a barrier and a device
    synchronisation on both sides, timed with events on that stream."""
    import torch
    if pre is not None:
        pre()
    torch.cuda.synchronize()
    _barrier(ws)
    with torch.cuda.stream(cs):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(cs)
        g.replay()
        e1.record(cs)
    torch.cuda.synchronize()
    _barrier(ws)
    return e0.elapsed_time(e1)


def _timed_replays(g, cs, ws, dev, min_ms, min_reps=3, max_reps=2000, pre=None):
    """Replays g (after one untimed replay) until about min_ms of timed work;
    every rank makes the same number of replays."""
    est = _max_over_ranks(_replay_ms(g, cs, ws, pre), ws, dev)
    reps = int(min(max_reps, max(min_reps, math.ceil(min_ms / max(est, 1e-3)))))
    return [_replay_ms(g, cs, ws, pre) for _ in range(reps)]


# --------------------------------------------------------------------------
# the oracle on the host cores
# --------------------------------------------------------------------------

def _threads_rate(work, nthreads, seconds):
    """work(t, i) -> units done (thread t, its i-th call; the oracle's C calls
    release the interpreter lock).  Every thread calls until `seconds` have
    passed; returns (units per second over the wall clock, units, wall s)."""
    counts = [0] * nthreads
    start = threading.Barrier(nthreads + 1)
    t_end = [0.0]

    def run(t):
        start.wait()
        i = 0
        while time.perf_counter() < t_end[0]:
            counts[t] += work(t, i)
            i += 1

    ths = [threading.Thread(target=run, args=(t,)) for t in range(nthreads)]
    for th in ths:
        th.start()
    t0 = time.perf_counter()
    t_end[0] = t0 + seconds
    start.wait()
    for th in ths:
        th.join()
    el = time.perf_counter() - t0
    return sum(counts) / el, sum(counts), el


def oracle_verify_rate(rows, drafts, T, seed, one_core_s, all_core_s, draft_logits=None,
                       seq_index=None):
    """The oracle's verification of a host sample (rows [n, K+1, V], drafts
    [n, K]) repeated over steps: seq-steps/s on one thread, then on every
    host core (each thread verifying the whole sample with its own steps)."""
    import oracle
    n = rows.shape[0]
    si = np.arange(n) if seq_index is None else seq_index

    def work(t, i):
        oracle.verify(rows, drafts, None, temperature=T, seed=seed, step=1000 * t + i,
                      draft_logits=draft_logits, seq_index=si)
        return n

    one, units1, el1 = _threads_rate(work, 1, one_core_s)
    nc = _nproc()
    alln, units_n, el_n = _threads_rate(work, nc, all_core_s)
    return {"one_core": round(one, 2), "all_cores": round(alln, 2), "nproc": nc,
            "ideal_all_cores": round(one * nc, 2),
            "sample": f"{n} sequences per call; one thread {units1} seq-steps in {el1:.2f} s, "
                      f"{nc} threads {units_n} seq-steps in {el_n:.2f} s"}


# --------------------------------------------------------------------------
# default line: verification at B=1024, K=3, bf16, T=1
# --------------------------------------------------------------------------

def head_config(ws, npool=HEAD_POOL):
    return {"workload": HEAD_WORKLOAD, "B_per_gpu": HEAD_B, "V": workloads.V_LARGE, "K": HEAD_K,
            "temperature": HEAD_T, "logits": "bf16 N(0, sd 2)",
            "drafts": "one-hot, each uniform among its row's top 5",
            "parallelism": f"dp{ws} (independent batches)",
            "l2": f"inputs larger than L2: {npool} rotating logits tensors of "
                  f"{HEAD_B * (HEAD_K + 1) * workloads.V_LARGE * 2 / 1e9:.2f} GB",
            "timing": "CUDA graph of exactly `steps` verify launches, replayed for >= "
                      f"{HEAD_MIN_TIMED_MS:.0f} ms; median replay; events on the capture stream"}


def run_verify_b1024(args, ws, rank, dev):
    import torch

    import sam_drafting_verification_gb300 as ss
    B, K, V, T = HEAD_B, HEAD_K, workloads.V_LARGE, HEAD_T
    steps, warm = args.steps, args.warmup
    hbm, peak_kind = _peaks()
    npool = max(1, args.pool)
    pool = [workloads.sweep_device(HEAD_SEED + 31 * i + 7919 * rank, B, K, V, torch.bfloat16, dev)
            for i in range(npool)]
    wsv = ss.verify_workspace(B, K, V, dev)
    res = {k: torch.empty(B, dtype=torch.int32, device=dev) for k in ("accept_len", "out_token", "status")}

    def step(s):
        lg, dr = pool[s % npool]
        ss.spec_verify(lg, dr, temperature=T, seed=HEAD_COIN_SEED, step=s, out=res, status=True,
                       workspace=wsv)

    for s in range(warm):
        step(s)
    torch.cuda.synchronize()
    g, cs = _capture(dev, lambda i: step(warm + i), steps)
    clocks = ClockSampler(dev.index or 0)
    clocks.start()
    time.sleep(0.3)
    times = _timed_replays(g, cs, ws, dev, HEAD_MIN_TIMED_MS)
    clk = clocks.stop()
    assert (res["status"] == 0).all(), "verification error"
    ms_step = _max_over_ranks(statistics.median(times) / steps, ws, dev)
    seqs = _sum_over_ranks(float(B), ws, dev)

    # rows each launch read (the chains' lengths): the same launches again, eagerly
    rows, acc = 0, 0
    for i in range(steps):
        step(warm + i)
        L = res["accept_len"].cpu().numpy().astype(np.int64)
        rows += int((L + 1).sum())
        acc += int(L.sum())
    alg = rows / steps * V * 2
    achieved = alg / (ms_step / 1e3) / 1e9
    roof = {"kernel": "verify_kernel<bf16, one-hot, T>0>", "bound": "hbm", "achieved": round(achieved, 1),
            "peak": hbm, "unit": "GB/s", "frac": round(achieved / hbm, 4),
            "traffic": _verify_traffic(HEAD_WORKLOAD),
            "peak_source": f"{peak_kind} hbm_gbs (burst copy)",
            "algorithmic_bytes_per_launch": round(alg, 1),
            "algorithmic_bytes": "sum over sequences of (accepted drafts + 1) rows x V x 2 B",
            "kernel_ms": round(ms_step, 5)}

    cpu = None
    if rank == 0:
        nb = 16
        host_rows = pool[0][0][:nb].float().cpu().numpy()
        host_dr = pool[0][1][:nb].cpu().numpy()
        c = oracle_verify_rate(host_rows, host_dr, T, HEAD_COIN_SEED, 10.0, 5.0)
        cpu = {"value": c["one_core"], "unit": "seq-steps/s", "cores": 1, "kind": "oracle",
               "nproc": c["nproc"], "all_cores": c["all_cores"], "ideal_all_cores": c["ideal_all_cores"],
               "sample": "fp64 verification of 16 sequences of the same workload (bf16 rows widened), "
                         + c["sample"]}
    e2e = e2e_verify(pool[:2] if npool > 1 else pool * 2, B, K, V, T, steps, dev)
    del pool
    torch.cuda.empty_cache()

    breakdown = {"verify_b1024": {"mean_accept": round(acc / (steps * B), 5),
                                  "rows_per_seq": round(rows / (steps * B), 5),
                                  "replays": len(times),
                                  "replay_ms_min_median_max": [round(min(times), 4),
                                                               round(statistics.median(times), 4),
                                                               round(max(times), 4)]}}
    if not args.no_breakdown:
        breakdown["step_b64"] = measure_step_b64(dev, ws, rank, cpu=rank == 0)
        torch.cuda.empty_cache()
        breakdown["sam_rollout_b256"] = measure_rollout(dev, ws, rank, cpu=rank == 0)
        torch.cuda.empty_cache()
        breakdown["draft_model_b32"] = measure_draft_model(dev, ws, rank, cpu=rank == 0)
        torch.cuda.empty_cache()
        breakdown["sweep_b1024"] = measure_sweep(dev, ws, rank)

    line = {
        "metric": METRIC, "value": round(seqs / (ms_step / 1e3), 1), "unit": "seq-steps/s", "n_gpus": ws,
        "steps": steps, "warmup": warm, "ms_per_step": round(ms_step, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32 (bf16 logits)", "data": "synthetic",
        "config": head_config(ws, npool),
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": len(times) * steps, "clocks": clk, "breakdown": breakdown,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def e2e_verify(pool, B, K, V, T, steps, dev):
    """The default line's metric through the public API with host buffers:
    every step copies its logits and drafts from pinned host memory, verifies
    and reads the accept lengths and emitted tokens back.  Step s + 1's copy
    runs on a copy stream into a second device buffer while step s verifies."""
    import torch

    import sam_drafting_verification_gb300 as ss
    host = [(pool[i][0].cpu().pin_memory(), pool[i][1].cpu().pin_memory()) for i in range(2)]
    dev_buf = [(torch.empty_like(pool[0][0]), torch.empty_like(pool[0][1])) for _ in range(2)]
    out = [{k: torch.empty(B, dtype=torch.int32, device=dev) for k in ("accept_len", "out_token", "status")}
           for _ in range(2)]
    h_acc = torch.empty((steps, B), dtype=torch.int32).pin_memory()
    h_tok = torch.empty((steps, B), dtype=torch.int32).pin_memory()
    wsv = ss.verify_workspace(B, K, V, dev)
    torch.cuda.synchronize()
    cur = torch.cuda.current_stream(dev)
    cps = torch.cuda.Stream(device=dev)
    copied = [torch.cuda.Event() for _ in range(2)]
    freed = [torch.cuda.Event() for _ in range(2)]

    def issue_copy(s):
        i = s % 2
        if s >= 2:  # the buffer's previous step has verified
            cps.wait_event(freed[i])
        with torch.cuda.stream(cps):
            dev_buf[i][0].copy_(host[s % 2][0], non_blocking=True)
            dev_buf[i][1].copy_(host[s % 2][1], non_blocking=True)
        copied[i].record(cps)

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(cur)
    cps.wait_stream(cur)
    issue_copy(0)
    for s in range(steps):
        if s + 1 < steps:
            issue_copy(s + 1)
        cur.wait_event(copied[s % 2])
        o = out[s % 2]
        ss.spec_verify(dev_buf[s % 2][0], dev_buf[s % 2][1], temperature=T, seed=HEAD_COIN_SEED, step=s,
                       out=o, status=True, workspace=wsv)
        freed[s % 2].record(cur)
        h_acc[s].copy_(o["accept_len"], non_blocking=True)
        h_tok[s].copy_(o["out_token"], non_blocking=True)
    e1.record(cur)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    assert (h_acc >= 0).all()
    h2d = int(dev_buf[0][0].numel() * 2 + dev_buf[0][1].numel() * 4)
    return {"value": round(B / (ms / 1e3), 1), "unit": "seq-steps/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": int(2 * B * 4),
            "ms_per_step": round(ms, 4), "steps": steps, "h2d_GBps": round(h2d / (ms / 1e3) / 1e9, 1),
            "overlap": "step s + 1's copy on a second stream while step s verifies"}


# --------------------------------------------------------------------------
# the full decode step at B=64 (automata + verification)
# --------------------------------------------------------------------------

def rs_inputs(rank: int, B: int = 64, V: int = workloads.V_LARGE, n: int = 4096, K: int = 3):
    """Histories and the continuation used to boost each pool entry's logits."""
    rng = np.random.default_rng(1002 + 7919 * rank)
    z = workloads.ZipfTokens(V, 1.1)
    streams = [workloads.make_stream(rng, n + POOL * (K + 1), V, 0.3, 8, 64, z) for _ in range(B)]
    hist = np.stack([s[:n] for s in streams]).astype(np.int32)
    cont = np.stack([s[n:] for s in streams]).astype(np.int32)  # [B, POOL*(K+1)]
    return hist, cont


def rs_logits_pool(device, B, K, V, cont, seed):
    """POOL bf16 tensors [B, K+1, V]: N(0, sd 2) plus 4 on the continuation."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    pool = []
    idx_b = torch.arange(B, device=device)
    for p in range(POOL):
        x = torch.empty((B, K + 1, V), dtype=torch.float32, device=device).normal_(0.0, 2.0, generator=g)
        truth = torch.as_tensor(cont[:, p * (K + 1):(p + 1) * (K + 1)], device=device).long()
        for j in range(K + 1):
            x[idx_b, j, truth[:, j]] += 4.0
        pool.append(x.to(torch.bfloat16).contiguous())
        del x
    return pool


class OracleLoop:
    """The oracle as it stands, on a sample of the B=64 workload: sequences
    [b0, b1) get their automata built over their histories (untimed); a step
    extends one with its previously emitted tokens, drafts K and verifies the
    draft in fp64 against that step's logits (host-generated, same
    distribution, bf16-rounded)."""

    def __init__(self, hist, cont, b0, b1, npool=4, seed=77):
        import oracle
        self.oracle = oracle
        V, K = workloads.V_LARGE, 3
        self.K, self.T, self.b0, self.b1, self.npool = K, 1.0, b0, b1, npool
        rng = np.random.default_rng(seed + b0)
        self.rows = []
        for p in range(npool):
            x = workloads.gaussian_logits(rng, (b1 - b0, K + 1, V), 2.0)
            workloads.boost_truth(x, cont[b0:b1, p * (K + 1):(p + 1) * (K + 1)], 4.0)
            self.rows.append(workloads.round_bf16(x))
        self.sams = [oracle.Sam(V) for _ in range(b1 - b0)]
        for i in range(b1 - b0):
            self.sams[i].extend(hist[b0 + i])
        self.emit = [[] for _ in range(b1 - b0)]

    def seq_step(self, i, s):
        K = self.K
        self.sams[i].extend(self.emit[i])
        d, dl, _, _ = self.sams[i].draft(K)
        d = np.maximum(d, 0)[None]
        rows = self.rows[s % self.npool][i:i + 1]
        r = self.oracle.verify(rows, d, np.array([dl], np.int32), temperature=self.T, seed=1002,
                               step=s, seq_index=np.array([self.b0 + i]))
        L = int(r["accept_len"][0])
        self.emit[i] = list(d[0, :L]) + [int(r["out_token"][0])]


def _step_worker(hist, cont, b0, b1, seconds, gate, q):
    """One host core's share of the oracle's B=64 decode steps (spawned
    process): builds its automata, waits at the gate, then steps its
    sequences until `seconds` have passed."""
    loop = OracleLoop(hist, cont, b0, b1)
    gate.wait()
    t_end = time.perf_counter() + seconds
    n, i = 0, 0
    while time.perf_counter() < t_end:
        for b in range(b1 - b0):
            loop.seq_step(b, i)
        n += b1 - b0
        i += 1
    q.put(n)


def oracle_step_rate(hist, cont, one_core_s, all_core_s):
    """Decode steps of the oracle on the B=64 workload: one thread over 16
    sequences, then one spawned process per host core, each with its own
    sequences."""
    import multiprocessing as mp
    nc = _nproc()
    one = OracleLoop(hist, cont, 0, 16)

    def w1(t, i):
        for b in range(16):
            one.seq_step(b, i)
        return 16

    r1, u1, el1 = _threads_rate(w1, 1, one_core_s)
    per = max(1, hist.shape[0] // nc)
    ctx = mp.get_context("spawn")
    gate = ctx.Barrier(nc + 1)
    q = ctx.Queue()
    procs = [ctx.Process(target=_step_worker,
                         args=(hist, cont, (t * per) % hist.shape[0], (t * per) % hist.shape[0] + per,
                               all_core_s, gate, q)) for t in range(nc)]
    for pr in procs:
        pr.start()
    gate.wait()
    t0 = time.perf_counter()
    un = sum(q.get(timeout=600) for _ in procs)
    eln = time.perf_counter() - t0
    for pr in procs:
        pr.join(timeout=60)
    rn = un / max(eln, all_core_s)
    return {"one_core": round(r1, 2), "all_cores": round(rn, 2), "nproc": nc,
            "ideal_all_cores": round(r1 * nc, 2),
            "sample": f"one thread: 16 sequences, {u1} seq-steps in {el1:.2f} s; {nc} processes x "
                      f"{per} sequences, {un} seq-steps in {eln:.2f} s (extend + draft + fp64 verify)"}


def measure_step_b64(dev, ws, rank, cpu=True, steps=64, warm=3, min_ms=300.0):
    """The full decode step at B=64: sam_step (extend by the previous step's
    emitted tokens, draft K=3), then spec_verify at T=1 on that step's
    logits; the emitted tokens feed the next step.  Verification is also
    timed alone on the drafts each step produced."""
    import torch

    import sam_drafting_verification_gb300 as ss
    B, V, K, T, n = 64, workloads.V_LARGE, 3, 1.0, 4096
    hist, cont = rs_inputs(rank, B, V, n, K)
    cap = n + (K + 1) * (steps + warm + 8) + 64
    batch = ss.SamBatch(B, cap, V, device=dev)
    hist_d = torch.as_tensor(hist, device=dev)
    nfull = torch.full((B,), n, dtype=torch.int32, device=dev)
    batch.extend(hist_d, nfull)  # untimed build, then the timed one
    torch.cuda.synchronize()
    batch.reset()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    batch.extend(hist_d, nfull)
    e1.record()
    torch.cuda.synchronize()
    prefill_ms = e0.elapsed_time(e1)
    assert (batch.status() == 0).all()
    snap = batch.export()
    pool = rs_logits_pool(dev, B, K, V, cont, 4242 + rank)
    emit = torch.zeros((B, K + 1), dtype=torch.int32, device=dev)
    emit_len = torch.zeros(B, dtype=torch.int32, device=dev)
    dlog = torch.empty((steps + warm, B, K), dtype=torch.int32, device=dev)
    llog = torch.empty((steps + warm, B), dtype=torch.int32, device=dev)
    aux = (torch.empty(B, dtype=torch.int32, device=dev), torch.empty(B, dtype=torch.int32, device=dev))
    out = {"accept_len": torch.empty(B, dtype=torch.int32, device=dev),
           "out_token": torch.empty(B, dtype=torch.int32, device=dev),
           "emit": emit, "emit_len": emit_len,
           "status": torch.empty(B, dtype=torch.int32, device=dev)}
    acc_log = torch.zeros((steps, B), dtype=torch.int32, device=dev)
    wsv = ss.verify_workspace(B, K, V, dev)

    def step(s, verify_only=False, log=False):
        if not verify_only:
            batch.step(emit, emit_len, K, out=(dlog[s], llog[s], aux[0], aux[1]))
        ss.spec_verify(pool[s % POOL], dlog[s], llog[s], temperature=T, seed=1002, step=s, out=out,
                       emit=True, status=True, workspace=wsv)
        if log:
            acc_log[s - warm].copy_(out["accept_len"])

    def restore():
        batch.import_(snap)
        emit_len.zero_()

    for s in range(warm):
        step(s)
    torch.cuda.synchronize()
    restore()
    g_full, cs = _capture(dev, lambda i: step(warm + i), steps)
    restore()
    # one eager pass of the same steps: accept lengths, and the drafts each
    # step produced (logged in dlog) for the verify-only graph
    for i in range(steps):
        step(warm + i, log=True)
    torch.cuda.synchronize()
    st_ok = bool((out["status"] == 0).all()) and bool((batch.status() == 0).all())
    g_ver, cs2 = _capture(dev, lambda i: step(warm + i, verify_only=True), steps)
    full = _timed_replays(g_full, cs, ws, dev, min_ms, pre=restore)
    ver = _timed_replays(g_ver, cs2, ws, dev, min_ms / 2)
    ms_full = _max_over_ranks(statistics.median(full) / steps, ws, dev)
    ms_ver = _max_over_ranks(statistics.median(ver) / steps, ws, dev)
    L = acc_log.cpu().numpy().astype(np.int64)
    hbm, _ = _peaks()
    vbytes = float((L + 1).sum()) / steps * V * 2
    r = {"B": B, "K": K, "V": V, "temperature": T, "history": n, "steps_per_replay": steps,
         "seq_steps_per_s": round(_sum_over_ranks(float(B), ws, dev) / (ms_full / 1e3), 1),
         "ms_per_step": round(ms_full, 5), "verify_us": round(ms_ver * 1e3, 2),
         "sam_ns_per_seq_step": round(max(ms_full - ms_ver, 0.0) * 1e6 / B, 1),
         "verify_frac_of_peak": round(vbytes / (ms_ver / 1e3) / 1e9 / hbm, 4),
         "verify_algorithmic_bytes_per_launch": round(vbytes, 1),
         "verify_traffic": _verify_traffic("rs_bf16_b64"),
         "mean_accept_len": round(float(L.mean()), 4),
         "prefill_tokens_per_s": round(B * n / (prefill_ms / 1e3), 1),
         "statuses_ok": st_ok}
    if cpu:
        c = oracle_step_rate(hist, cont, 5.0, 4.0)
        r["oracle_seq_steps_per_s"] = c
        r["vs_oracle_one_core"] = round(r["seq_steps_per_s"] / c["one_core"], 1)
        r["vs_oracle_all_cores"] = round(r["seq_steps_per_s"] / c["all_cores"], 1)
    return r


def run_rs(args, ws, rank, dev):
    r = measure_step_b64(dev, ws, rank, cpu=rank == 0, steps=args.steps, warm=args.warmup)
    hbm, peak_kind = _peaks()
    c = r.get("oracle_seq_steps_per_s")
    ver_ms = r["verify_us"] / 1e3
    line = {"metric": METRIC, "value": r["seq_steps_per_s"], "unit": "seq-steps/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32 (bf16 logits)", "data": "synthetic",
            "config": {"workload": "rs_bf16_b64", "B_per_gpu": 64, "V": r["V"], "K": 3, "temperature": 1.0,
                       "history": 4096, "logits": "bf16 N(0, sd 2) + 4 on the true continuation",
                       "drafts": "device SAM (K=3)", "l2": f"rotating pool of {POOL} logits tensors",
                       "timing": "CUDA graph of exactly `steps` steps, median replay"},
            "roofline": {"kernel": "verify_kernel<bf16, one-hot, T>0>", "bound": "hbm",
                         "achieved": round(r["verify_algorithmic_bytes_per_launch"] / ver_ms / 1e6, 1),
                         "peak": hbm, "unit": "GB/s", "frac": r["verify_frac_of_peak"],
                         "traffic": r["verify_traffic"], "peak_source": peak_kind,
                         "algorithmic_bytes_per_launch": r["verify_algorithmic_bytes_per_launch"]},
            "cpu_baseline": ({"value": c["one_core"], "unit": "seq-steps/s", "cores": 1, "kind": "oracle",
                              "nproc": c["nproc"], "all_cores": c["all_cores"], "sample": c["sample"]}
                             if c else None),
            "gpu_launches": 2 * args.steps, "breakdown": r}
    if rank == 0:
        print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------
# the automata alone: long-tail rollout, B=256 histories of 16k-32k tokens
# --------------------------------------------------------------------------

def _rollout_inputs(rank):
    w = workloads.long_rollout(seed=1004 + 7919 * rank)
    B, steps = w["B"], w["steps"]
    lens, n_new, streams = w["lens"], w["n_new"], w["streams"]
    maxlen = int(lens.max())
    pre = np.zeros((B, maxlen), np.int32)
    toks = np.zeros((steps, B, 4), np.int32)
    for b in range(B):
        pre[b, :lens[b]] = streams[b][:lens[b]]
        pos = int(lens[b])
        for s in range(steps):
            k = int(n_new[s, b])
            toks[s, b, :k] = streams[b][pos:pos + k]
            pos += k
    return w, pre, toks


def _rollout_worker(hists, toks, n_new, K, gate, q):
    """One host core's share of the oracle's rollout (spawned process):
    builds its automata over `hists` between two gates, then runs every step
    of extend + draft between the next two."""
    import oracle
    V = workloads.V_LARGE
    sams = [oracle.Sam(V) for _ in hists]
    toks = np.ascontiguousarray(toks)
    n_new = np.ascontiguousarray(n_new)
    gate.wait()
    t0 = time.perf_counter()
    for i, h in enumerate(hists):
        sams[i].extend(h)
    t1 = time.perf_counter()
    gate.wait()
    t2 = time.perf_counter()
    for s in range(toks.shape[0]):
        oracle.step_batch(sams, toks[s], n_new[s], K)
    t3 = time.perf_counter()
    gate.wait()
    q.put((t1 - t0, t3 - t2))


def oracle_rollout_rates(streams, lens, toks, n_new, K, one_core_seqs=32):
    """The oracle's automata on samples of the rollout: the prefill build
    (tokens/s) and 512 steps of extend + draft (ns per sequence-step), on
    one thread over `one_core_seqs` sequences, then on every host core (one
    spawned process each, with as many sequences)."""
    import multiprocessing as mp

    import oracle
    V = workloads.V_LARGE
    nc = _nproc()
    steps = toks.shape[0]
    B = len(lens)
    per = one_core_seqs
    seqs1 = list(range(per))
    sams = [oracle.Sam(V) for _ in seqs1]
    t0 = time.perf_counter()
    for i, b in enumerate(seqs1):
        sams[i].extend(streams[b][:lens[b]])
    b1 = time.perf_counter() - t0
    tk1 = np.ascontiguousarray(toks[:, seqs1])
    nn1 = np.ascontiguousarray(n_new[:, seqs1])
    t0 = time.perf_counter()
    for s in range(steps):
        oracle.step_batch(sams, tk1[s], nn1[s], K)
    s1 = time.perf_counter() - t0
    tok1 = int(sum(int(lens[b]) for b in seqs1))
    del sams
    groups = [[(t * per + i) % B for i in range(per)] for t in range(nc)]
    ctx = mp.get_context("spawn")
    gate = ctx.Barrier(nc + 1)
    q = ctx.Queue()
    procs = [ctx.Process(target=_rollout_worker,
                         args=([streams[b][:lens[b]] for b in g], toks[:, g], n_new[:, g], K, gate, q))
             for g in groups]
    for pr in procs:
        pr.start()
    gate.wait()
    w0 = time.perf_counter()
    gate.wait()
    w1 = time.perf_counter()
    gate.wait()
    w2 = time.perf_counter()
    per_proc = [q.get(timeout=600) for _ in procs]
    for pr in procs:
        pr.join(timeout=60)
    bn, sn = w1 - w0, w2 - w1
    tokn = int(sum(int(lens[b]) for g in groups for b in g))
    return {"nproc": nc,
            "prefill_tokens_per_s": {"one_core": round(tok1 / b1, 1), "all_cores": round(tokn / bn, 1),
                                     "ideal_all_cores": round(tok1 / b1 * nc, 1)},
            "ns_per_seq_step": {"one_core": round(s1 / (steps * per) * 1e9, 1),
                                "all_cores": round(sn / (steps * per * nc) * 1e9, 1),
                                "ideal_all_cores": round(s1 / (steps * per) * 1e9 / nc, 1)},
            "sample": f"one thread: {per} sequences ({tok1} history tokens, build {b1:.2f} s, "
                      f"{steps} steps {s1:.3f} s); {nc} processes x {per} sequences ({tokn} tokens, "
                      f"build {bn:.2f} s, steps {sn:.3f} s; slowest process build "
                      f"{max(x[0] for x in per_proc):.2f} s, steps {max(x[1] for x in per_proc):.3f} s)"}


def measure_rollout(dev, ws, rank, cpu=True, min_ms=400.0):
    """B=256 histories log-uniform in [16k, 32k] tokens (Zipf(1.1), copy prob
    0.5, spans 16-256), V=151936: the prefill build, then 512 steps of
    (extend by the stream's next U{1..4} tokens + draft K=3), timed alone and
    with greedy verification of bf16 logits N(0, sd 2) [256, 4, V]."""
    import torch

    import sam_drafting_verification_gb300 as ss
    w, pre, toks = _rollout_inputs(rank)
    B, V, K, steps = w["B"], w["V"], w["K"], w["steps"]
    lens, n_new, streams = w["lens"], w["n_new"], w["streams"]
    cap = int(max(len(x) for x in streams))
    batch = ss.SamBatch(B, cap, V, device=dev)
    pre_d = torch.as_tensor(pre, device=dev)
    lens_d = torch.as_tensor(lens, device=dev)
    toks_d = torch.as_tensor(toks, device=dev)
    nn_d = torch.as_tensor(n_new, device=dev)
    batch.extend(pre_d, lens_d)
    torch.cuda.synchronize()
    batch.reset()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    batch.extend(pre_d, lens_d)
    e1.record()
    torch.cuda.synchronize()
    prefill_ms = e0.elapsed_time(e1)
    assert (batch.status() == 0).all()
    snap = batch.export()
    npool = 4
    g = torch.Generator(device=dev)
    g.manual_seed(4004 + rank)
    pool = []
    for _ in range(npool):
        x = torch.empty((B, K + 1, V), dtype=torch.bfloat16, device=dev)
        for b0 in range(0, B, 64):
            x[b0:b0 + 64] = torch.empty((min(64, B - b0), K + 1, V), device=dev).normal_(0.0, 2.0, generator=g)
        pool.append(x)
    draft = torch.empty((B, K), dtype=torch.int32, device=dev)
    dlen = torch.empty(B, dtype=torch.int32, device=dev)
    mlen = torch.empty(B, dtype=torch.int32, device=dev)
    mend = torch.empty(B, dtype=torch.int32, device=dev)
    out = {"accept_len": torch.empty(B, dtype=torch.int32, device=dev),
           "out_token": torch.empty(B, dtype=torch.int32, device=dev),
           "status": torch.empty(B, dtype=torch.int32, device=dev)}
    wsv = ss.verify_workspace(B, K, V, dev)

    def step(s, verify=True):
        batch.step(toks_d[s], nn_d[s], K, out=(draft, dlen, mlen, mend))
        if verify:
            ss.spec_verify(pool[s % npool], draft, dlen, temperature=0.0, out=out, status=True,
                           workspace=wsv)

    def restore():
        batch.import_(snap)

    for s in range(3):
        step(s)
    torch.cuda.synchronize()
    restore()
    g_full, cs1 = _capture(dev, lambda s: step(s), steps)
    g_sam, cs2 = _capture(dev, lambda s: step(s, verify=False), steps)
    full = _timed_replays(g_full, cs1, ws, dev, min_ms, pre=restore)
    sam = _timed_replays(g_sam, cs2, ws, dev, min_ms, pre=restore)
    assert (out["status"].cpu() == 0).all() and (batch.status() == 0).all()
    # the automata followed the streams: the last drafts equal a fresh query
    st_ms = _max_over_ranks(statistics.median(full) / steps, ws, dev)
    sam_ns = _max_over_ranks(statistics.median(sam) / steps / B * 1e6, ws, dev)
    r = {"B": B, "K": K, "V": V, "steps": steps, "prefill_tokens": int(lens.sum()),
         "sam_ns_per_seq_step": round(sam_ns, 1),
         "step_with_greedy_verify_us": round(st_ms * 1e3, 2),
         "seq_steps_per_s_with_verify": round(_sum_over_ranks(float(B), ws, dev) / (st_ms / 1e3), 1),
         "prefill_tokens_per_s": round(float(lens.sum()) / (prefill_ms / 1e3), 1),
         "prefill_ms": round(prefill_ms, 3),
         "replays": [len(full), len(sam)]}
    if cpu:
        c = oracle_rollout_rates(streams, lens, toks, n_new, K)
        r["oracle"] = c
        r["sam_vs_oracle_one_core"] = round(c["ns_per_seq_step"]["one_core"] / sam_ns, 1)
        r["sam_vs_oracle_all_cores"] = round(c["ns_per_seq_step"]["all_cores"] / sam_ns, 1)
        r["prefill_vs_oracle_one_core"] = round(r["prefill_tokens_per_s"] / c["prefill_tokens_per_s"]["one_core"], 1)
        r["prefill_vs_oracle_all_cores"] = round(r["prefill_tokens_per_s"] / c["prefill_tokens_per_s"]["all_cores"], 1)
    return r


def run_rollout(args, ws, rank, dev):
    r = measure_rollout(dev, ws, rank, cpu=rank == 0)
    c = r.get("oracle")
    line = {"metric": METRIC, "value": r["sam_ns_per_seq_step"], "unit": "ns/seq-step (SAM extend + draft)",
            "n_gpus": ws, "steps": r["steps"], "warmup": 3,
            "ms_per_step": round(r["sam_ns_per_seq_step"] * r["B"] / 1e6, 5),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "int32",
            "data": "synthetic",
            "config": {"workload": "long_rollout_b256", "B_per_gpu": r["B"], "V": r["V"], "K": r["K"],
                       "steps": r["steps"], "history": "log-uniform [16384, 32768]",
                       "prefill_tokens": r["prefill_tokens"],
                       "timing": "CUDA graph of the 512 SAM steps, median replay"},
            "cpu_baseline": ({"value": c["ns_per_seq_step"]["one_core"], "unit": "ns/seq-step", "cores": 1,
                              "kind": "oracle", "nproc": c["nproc"],
                              "all_cores": c["ns_per_seq_step"]["all_cores"], "sample": c["sample"]}
                             if c else None),
            "gpu_launches": r["steps"], "breakdown": r}
    if rank == 0:
        print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------
# verification with draft-model logits: B=32, K=5, fp32, T=0.7
# --------------------------------------------------------------------------

DM_POOL = 4


def measure_draft_model(dev, ws, rank, cpu=True, reps=20, min_ms=200.0):
    """Target N(0, sd 2) [32, 6, V] fp32, draft logits = target + N(0, 1)
    [32, 5, V] fp32, drafts sampled from softmax(draft / 0.7), T=0.7:
    accept with min(1, p/q), resample from norm(max(0, p - q)).  Four input
    sets rotate (856 MB).  Algorithmic bytes of a launch: per sequence the
    (L + 1) target rows and min(L + 1, n) draft rows its chain scored, plus
    one residual pass over the final target and draft rows after a
    rejection."""
    import torch

    import sam_drafting_verification_gb300 as ss
    B, K, V, T = 32, 5, workloads.V_LARGE, 0.7
    hbm, peak_kind = _peaks()
    pool = [workloads.draft_model_device(1003 + 17 * i + 7919 * rank, B, K, V, T, dev) for i in range(DM_POOL)]
    wsv = ss.verify_workspace(B, K, V, dev)
    res = {k: torch.empty(B, dtype=torch.int32, device=dev) for k in ("accept_len", "out_token", "status")}

    def step(s):
        tg, dl, dr = pool[s % DM_POOL]
        ss.spec_verify(tg, dr, draft_logits=dl, temperature=T, seed=3, step=s, out=res, status=True,
                       workspace=wsv)

    for s in range(3):
        step(s)
    torch.cuda.synchronize()
    g, cs = _capture(dev, step, reps)
    times = _timed_replays(g, cs, ws, dev, min_ms)
    ms = _max_over_ranks(statistics.median(times) / reps, ws, dev)
    acc, rows_t, rows_d, resid = 0, 0, 0, 0
    for s in range(reps):
        step(s)
        L = res["accept_len"].cpu().numpy().astype(np.int64)
        assert (res["status"] == 0).all()
        acc += int(L.sum())
        rows_t += int((L + 1).sum())
        rows_d += int(np.minimum(L + 1, K).sum())
        resid += int((L < K).sum())
    alg = (rows_t + rows_d + 2 * resid) / reps * V * 4
    ach = alg / (ms / 1e3) / 1e9
    r = {"B": B, "K": K, "V": V, "temperature": T, "us_per_launch": round(ms * 1e3, 2),
         "seq_steps_per_s": round(_sum_over_ranks(float(B), ws, dev) / (ms / 1e3), 1),
         "acceptance": round(acc / (reps * B * K), 4), "mean_accept_len": round(acc / (reps * B), 4),
         "algorithmic_bytes_per_launch": round(alg, 1), "achieved_GBps": round(ach, 1),
         "frac": round(ach / hbm, 4), "peak_source": peak_kind,
         "traffic": _verify_traffic("draft_model_b32")}
    if cpu:
        nb = 4
        tg, dl, dr = pool[0]
        c = oracle_verify_rate(tg[:nb].cpu().numpy(), dr[:nb].cpu().numpy(), T, 3, 5.0, 4.0,
                               draft_logits=dl[:nb].cpu().numpy())
        r["oracle_seq_steps_per_s"] = c
    return r


def run_draft_model(args, ws, rank, dev):
    r = measure_draft_model(dev, ws, rank, cpu=rank == 0, reps=args.steps)
    hbm, peak_kind = _peaks()
    c = r.get("oracle_seq_steps_per_s")
    line = {"metric": METRIC, "value": r["seq_steps_per_s"], "unit": "seq-steps/s", "n_gpus": ws,
            "steps": args.steps, "warmup": 3, "ms_per_step": round(r["us_per_launch"] / 1e3, 6),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": "draft_model_b32", "B_per_gpu": r["B"], "V": r["V"], "K": r["K"],
                       "temperature": r["temperature"], "logits": "fp32 target N(0, sd 2), draft = target + N(0, 1)",
                       "drafts": "sampled from softmax(draft / 0.7)", "l2": f"{DM_POOL} rotating input sets (856 MB)",
                       "timing": "CUDA graph of `steps` launches, median replay"},
            "roofline": {"kernel": "verify_kernel<f32, f32 draft logits, T>0>", "bound": "hbm",
                         "achieved": r["achieved_GBps"], "peak": hbm, "unit": "GB/s", "frac": r["frac"],
                         "traffic": r["traffic"], "peak_source": peak_kind,
                         "algorithmic_bytes_per_launch": r["algorithmic_bytes_per_launch"]},
            "cpu_baseline": ({"value": c["one_core"], "unit": "seq-steps/s", "cores": 1, "kind": "oracle",
                              "nproc": c["nproc"], "all_cores": c["all_cores"], "sample": c["sample"]}
                             if c else None),
            "gpu_launches": args.steps, "breakdown": r}
    if rank == 0:
        print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------
# verification sweep at B=1024
# --------------------------------------------------------------------------

def measure_sweep(dev, ws, rank, reps=10, only=None):
    """B=1024, V=151936, K in {1,3,5,8} x fp32/bf16 x {greedy, T=1, greedy
    with drafts = each row's argmax (every row read)}; logits N(0, sd 2),
    drafts uniform among each row's top 5.  Each point: a graph of `reps`
    launches on one input (above L2 at every point: each launch reads at
    least 1024 rows), median of three replays."""
    import torch

    import sam_drafting_verification_gb300 as ss
    B, V = 1024, workloads.V_LARGE
    hbm, _ = _peaks()
    points = []
    for K in (1, 3, 5, 8):
        for dtype in (torch.float32, torch.bfloat16):
            if only and (only[0] != K or only[1] != dtype):
                continue
            logits, draft = workloads.sweep_device(7000 + K + 100 * rank, B, K, V, dtype, dev)
            full_draft = torch.argmax(logits[:, :K].float(), dim=-1).to(torch.int32).contiguous()
            for T, name, dr in ((0.0, "greedy", draft), (1.0, "T=1", draft), (0.0, "greedy-full-read", full_draft)):
                if only and only[2] != name:
                    continue
                wsv = ss.verify_workspace(B, K, V, dev)
                res = ss.spec_verify(logits, dr, None, temperature=T, seed=5, step=0, workspace=wsv)
                for w in range(3):
                    ss.spec_verify(logits, dr, None, temperature=T, seed=5, step=w, out=res, workspace=wsv)
                torch.cuda.synchronize()
                g, cs = _capture(dev, lambda r: ss.spec_verify(logits, dr, None, temperature=T, seed=5, step=r,
                                                               out=res, workspace=wsv), reps)
                times = [_replay_ms(g, cs, ws) for _ in range(4)][1:]
                ms = _max_over_ranks(statistics.median(times) / reps, ws, dev)
                Lh = res["accept_len"].cpu().numpy().astype(np.int64)
                alg = float((Lh + 1).sum()) * V * logits.element_size()
                points.append({"K": K, "dtype": str(dtype).split(".")[-1], "mode": name,
                               "us": round(ms * 1e3, 2), "seq_steps_per_s": round(B / (ms / 1e3), 1),
                               "mean_accept": round(float(Lh.mean()), 4),
                               "alg_GBps": round(alg / (ms / 1e3) / 1e9, 1),
                               "frac": round(alg / (ms / 1e3) / 1e9 / hbm, 4)})
                del g
            del logits, draft, full_draft
            torch.cuda.empty_cache()
    return points


def run_sweep(args, ws, rank, dev):
    import torch
    only = None
    if args.point:  # "K,dtype,mode", e.g. "3,bf16,T=1": one sweep point (profiling)
        k_s, d_s, m_s = args.point.split(",")
        only = (int(k_s), {"f32": torch.float32, "bf16": torch.bfloat16}[d_s], m_s)
    hbm, peak_kind = _peaks()
    points = measure_sweep(dev, ws, rank, reps=max(args.steps, 1), only=only)
    head = points[0]
    for p in points:  # the default line's point when present
        if (p["K"], p["dtype"], p["mode"]) == (HEAD_K, "bfloat16", "T=1"):
            head = p
    line = {"metric": METRIC, "value": head["seq_steps_per_s"], "unit": "seq-steps/s", "n_gpus": ws,
            "steps": args.steps, "warmup": 3, "ms_per_step": head["us"] / 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": "sweep_b1024", "B": 1024, "V": workloads.V_LARGE,
                       "point": {k: head[k] for k in ("K", "dtype", "mode")}},
            "roofline": {"bound": "hbm", "achieved": head["alg_GBps"], "peak": hbm, "unit": "GB/s",
                         "frac": head["frac"], "traffic": None, "peak_source": peak_kind},
            "points": points}
    if rank == 0:
        print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------
# toy-model rollout: the decode loop end to end, with and without speculation
# --------------------------------------------------------------------------

class ToyTarget:
    """Stand-in for the target model: logits at (sequence b, new-token index p)
    are a row of a seeded N(0, sd 2) pool plus `boost` on the stream's true
    token, so greedy decoding reproduces the stream (Zipf tokens with copied
    spans) and SAM drafts are accepted where the stream repeats itself."""

    def __init__(self, truth, V, boost, dev, dtype, P=127, seed=4004):
        import torch
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        self.noise = torch.empty((P, V), device=dev).normal_(0.0, 2.0, generator=g)
        self.truth = torch.as_tensor(truth, dtype=torch.int64, device=dev)
        self.boost, self.P, self.V, self.dtype = boost, P, V, dtype

    def __call__(self, rows, n_done, draft, draft_len):
        import torch
        n, K = draft.shape
        r = rows.long().repeat_interleave(K + 1)
        p = (n_done.view(-1, 1) + torch.arange(K + 1, device=rows.device).view(1, -1)).reshape(-1)
        x = self.noise[(r * 7919 + p) % self.P]
        t = self.truth[r, p.clamp(max=self.truth.shape[1] - 1)]
        x[torch.arange(x.shape[0], device=x.device), t] += self.boost
        return x.to(self.dtype).view(n, K + 1, self.V).contiguous()


def run_rollout_toy(args, ws, rank, dev):
    """B=64 sequences with 4096-token Zipf(1.1) prompts (copy prob 0.3, spans
    8-64) generating log-uniform [64, 1024] new tokens each (a long tail),
    V=151936, bf16 logits from ToyTarget, greedy.  Three loops over the same
    inputs: plain decoding (K=0), speculation at every step (K=3), and the
    adaptive switch (K=3 only while at most 8 sequences are active).  Each
    loop's tokens must equal the streams (lossless)."""
    import torch

    import sam_drafting_verification_gb300 as ss
    from sam_drafting_verification_gb300.rollout import Rollout
    B, V, K, n0, thr = 64, workloads.V_LARGE, 3, 4096, 8
    rng = np.random.default_rng(1005 + 7919 * rank)
    limits = workloads.log_uniform_lengths(rng, B, 64, 1024).astype(np.int64)
    z = workloads.ZipfTokens(V, 1.1)
    streams = [workloads.make_stream(rng, n0 + int(limits.max()) + 8, V, 0.3, 8, 64, z) for _ in range(B)]
    prompts = np.stack([s[:n0] for s in streams]).astype(np.int32)
    truth = np.stack([s[n0:] for s in streams]).astype(np.int64)
    model = ToyTarget(truth, V, 40.0, dev, torch.bfloat16)
    modes = {}
    for name, k, t in (("plain", 0, None), ("speculate", K, None), ("adaptive", K, thr)):
        batch = ss.SamBatch(B, n0 + int(limits.max()) + 64, V, device=dev)
        batch.extend(torch.as_tensor(prompts, device=dev), torch.full((B,), n0, dtype=torch.int32, device=dev))
        Rollout(batch, model, K=k, threshold=t).run(np.minimum(limits, 16))  # warm-up
        batch.reset()
        batch.extend(torch.as_tensor(prompts, device=dev), torch.full((B,), n0, dtype=torch.int32, device=dev))
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        res = Rollout(batch, model, K=k, threshold=t).run(limits)
        torch.cuda.synchronize()
        el = time.perf_counter() - t0
        ok = all(res.tokens[b] == truth[b, :limits[b]].tolist() for b in range(B))
        assert ok, f"{name}: rollout differs from plain decoding"
        ntok = int(limits.sum())
        modes[name] = {"steps": res.steps, "tokens": ntok, "seconds": round(el, 4),
                       "tokens_per_s": round(ntok / el, 1),
                       "tokens_per_step": round(ntok / res.steps, 3),
                       "accepted_drafts": res.accepted,
                       "speculative_steps": sum(1 for x in res.k_per_step if x > 0)}
    line = {"metric": "generated tokens/s, toy-model rollout (decode loop through sam_spec_step)",
            "value": modes["speculate"]["tokens_per_s"], "unit": "tokens/s", "n_gpus": ws,
            "steps": modes["speculate"]["steps"], "warmup": 1, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32 (bf16 logits)",
            "data": "synthetic",
            "config": {"workload": "rollout_toy_b64", "B": B, "V": V, "K": K, "threshold": thr,
                       "prompt": n0, "new_tokens": "log-uniform [64, 1024] per sequence",
                       "target": "ToyTarget (seeded noise + 40 on the stream token), greedy",
                       "timing": "wall clock of the whole loop, host bookkeeping and the toy "
                                 "model's logits included"},
            "modes": modes,
            "lossless": True}
    if rank == 0:
        print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------
# static corpus automaton: build and matching
# --------------------------------------------------------------------------

def run_static_match(args, ws, rank, dev):
    """A corpus of ~1M tokens (documents of 200-4000 Zipf(1.1) tokens with
    copied spans, V=151936, joined by an end-of-sequence token) built once on
    the device; 256 generated texts (corpus passages of 16-256 tokens with
    1-8 fresh tokens between them) followed 1-4 tokens per step for 512 steps
    with K=3 corpus drafts, in one CUDA graph.  Reports the build rate and ns
    per sequence-step of the matching, next to the oracle's matching of the
    same texts on one host core."""
    import torch

    import oracle
    import sam_drafting_verification_gb300 as ss
    V, B, K, steps = workloads.V_LARGE, 256, 3, 512
    eos = V - 1
    rng = np.random.default_rng(1006 + 7919 * rank)
    z = workloads.ZipfTokens(V, 1.1)
    docs, total = [], 0
    while total < 1_000_000:
        d = workloads.make_stream(rng, int(rng.integers(200, 4000)), V, 0.3, 8, 64, z)
        docs.append(np.concatenate([d, [eos]]))
        total += len(docs[-1])
    corpus = np.concatenate(docs).astype(np.int32)
    n_new = rng.integers(1, 5, size=(steps, B)).astype(np.int32)
    need = n_new.sum(axis=0)
    gens = []
    for b in range(B):
        parts, n = [], 0
        while n < need[b]:
            a = int(rng.integers(0, len(corpus) - 300))
            parts.append(corpus[a:a + int(rng.integers(16, 257))])
            parts.append(z.draw(rng, int(rng.integers(1, 9))))
            n += len(parts[-2]) + len(parts[-1])
        gens.append(np.concatenate(parts)[:need[b]].astype(np.int32))
    toks = np.zeros((steps, B, 4), np.int32)
    for b in range(B):
        pos = 0
        for s in range(steps):
            k = int(n_new[s, b])
            toks[s, b, :k] = gens[b][pos:pos + k]
            pos += k
    cb = ss.SamBatch(1, len(corpus), V, device=dev)
    cd = torch.as_tensor(corpus[None, :], device=dev)
    cl = torch.tensor([len(corpus)], dtype=torch.int32, device=dev)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    cb.extend(cd, cl)
    torch.cuda.synchronize()
    build_s = time.perf_counter() - t0
    assert cb.status()[0] == 0
    state = torch.zeros((B, 2), dtype=torch.int32, device=dev)
    td = torch.as_tensor(toks, device=dev)
    nd = torch.as_tensor(n_new, device=dev)
    outs = tuple(torch.empty(sz, dtype=torch.int32, device=dev) for sz in ((B, K), (B,), (B,), (B,)))
    for s in range(3):  # warm-up
        cb.match(0, state, td[s], nd[s], K, out=outs)
    torch.cuda.synchronize()
    cs = torch.cuda.Stream(device=dev)
    g = torch.cuda.CUDAGraph()
    cs.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(cs):
        with torch.cuda.graph(g, stream=cs):
            for s in range(steps):
                cb.match(0, state, td[s], nd[s], K, out=outs)
    torch.cuda.synchronize()
    state.zero_()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    g.replay()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    ns_gpu = ms * 1e6 / (steps * B)
    # the oracle on the same texts (corpus built untimed)
    cpu = None
    if rank == 0:
        osam = oracle.Sam(V)
        osam.extend(corpus)
        ost = np.zeros((B, 2), np.int32)
        t0 = time.perf_counter()
        for s in range(steps):
            oracle.match_batch(osam, ost, toks[s], n_new[s], K)
        el = time.perf_counter() - t0
        assert np.array_equal(ost, state.cpu().numpy()), "device and oracle matching states differ"
        ns_cpu = el / (steps * B) * 1e9
        cpu = {"value": round(ns_cpu, 1), "unit": "ns/seq-step (static matching + draft)", "cores": 1,
               "kind": "oracle", "sample": f"the same {B} texts x {steps} steps, one C call per step "
                                            f"for all {B} texts, {el:.2f} s"}
    line = {"metric": "static-automaton matching ns/seq-step (K=3 corpus drafts)",
            "value": round(ns_gpu, 2), "unit": "ns/seq-step", "n_gpus": ws, "steps": steps,
            "warmup": 3, "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
            "dtype": "int32", "data": "synthetic",
            "config": {"workload": "static_match_b256", "corpus_tokens": int(len(corpus)),
                       "documents": len(docs), "B": B, "K": K, "V": V,
                       "timing": "CUDA graph of the 512 matching launches"},
            "cpu_baseline": cpu,
            "breakdown": {"corpus_build_tokens_per_s": round(len(corpus) / build_s, 1),
                          "corpus_build_s": round(build_s, 3),
                          "speedup_vs_oracle": (round(cpu["value"] / ns_gpu, 1) if cpu else None)}}
    if rank == 0:
        print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------
# tree-draft verification
# --------------------------------------------------------------------------

# node n's parent: a root with three candidates (nodes 1, 4, 7); nodes 1 and
# 4 each carry a chain of two more drafts
TREE_PARENT = (-1, 0, 1, 2, 0, 4, 5, 0)
TREE_BOOST = (0.0, 14.0, 14.0, 14.0, 12.0, 12.0, 12.0, 11.0)
TREE_REPLAYS = 10


def tree_arrays(rng, B, V):
    """tok / first_child / next_sibling [B, 8] of the fixed tree shape, with
    random tokens (distinct among siblings)."""
    N = len(TREE_PARENT)
    fc = np.full(N, -1, np.int32)
    ns = np.full(N, -1, np.int32)
    last = {}
    for n in range(1, N):
        p = TREE_PARENT[n]
        if p in last:
            ns[last[p]] = n
        else:
            fc[p] = n
        last[p] = n
    tok = np.full((B, N), -1, np.int32)
    for b in range(B):
        t = rng.choice(V, N - 1, replace=False)
        tok[b, 1:] = t
    return tok, np.tile(fc, (B, 1)), np.tile(ns, (B, 1))


def run_tree(args, ws, rank, dev):
    """B=256 draft trees of 8 nodes (three candidates under the root, two of
    them with chains of two more: up to 3 accepted drafts), V=151936, bf16
    logits N(0, sd 2) with each node's token raised in its parent's row by
    14 / 12 / 11 (first / second / third candidate branch), rejection sampling
    at T=1.  Two step tensors of 622 MB alternate (each far above L2); the
    timed region replays a CUDA graph of the verify launches ten times.  Algorithmic
    bytes per launch: the rows the walk reads, sum over sequences of
    (accepted depth + 1) x V x 2."""
    import torch

    import oracle
    import sam_drafting_verification_gb300 as ss
    B, V, T = 256, workloads.V_LARGE, 1.0
    N = len(TREE_PARENT)
    reps = min(max(args.steps, 1), 1000)
    hbm, peak_kind = _peaks()
    rng = np.random.default_rng(1007 + 7919 * rank)
    pool = []
    trees = []
    for i in range(2):
        tok, fc, ns = tree_arrays(rng, B, V)
        g = torch.Generator(device=dev)
        g.manual_seed(5000 + 31 * i + 7919 * rank)
        lg = torch.empty((B, N, V), dtype=torch.bfloat16, device=dev)
        for b0 in range(0, B, 64):
            x = torch.empty((min(64, B - b0), N, V), dtype=torch.float32, device=dev).normal_(0.0, 2.0, generator=g)
            lg[b0:b0 + 64] = x.to(torch.bfloat16)
        par = np.array(TREE_PARENT[1:])
        bb = np.repeat(np.arange(B), N - 1)
        rows = np.tile(par, B)
        cols = tok[:, 1:].reshape(-1)
        boost = torch.tensor(np.tile(TREE_BOOST[1:], B), dtype=torch.float32, device=dev)
        idx = tuple(torch.as_tensor(a, device=dev) for a in (bb, rows, cols))
        lg.index_put_(idx, (lg[idx].float() + boost).to(torch.bfloat16))
        pool.append(lg)
        trees.append(tuple(torch.as_tensor(a, device=dev) for a in (tok, fc, ns)))
    wsv = ss.verify_workspace(B, N - 1, V, dev)
    res = ss.spec_verify_tree(pool[0], *trees[0], temperature=T, seed=11, step=0, workspace=wsv)
    for w in range(max(args.warmup, 3)):
        ss.spec_verify_tree(pool[w % 2], *trees[w % 2], temperature=T, seed=11, step=w, workspace=wsv, out=res)
    torch.cuda.synchronize()
    cs = torch.cuda.Stream(device=dev)
    graph = torch.cuda.CUDAGraph()
    cs.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(cs):
        with torch.cuda.graph(graph, stream=cs):
            for r in range(reps):
                ss.spec_verify_tree(pool[r % 2], *trees[r % 2], temperature=T, seed=11, step=r,
                                    workspace=wsv, out=res)
    torch.cuda.synchronize()
    clk = ClockSampler(dev.index or 0)
    clk.start()
    _barrier(ws)
    torch.cuda.synchronize()
    with torch.cuda.stream(cs):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(cs)
        for _ in range(TREE_REPLAYS):
            graph.replay()
        e1.record(cs)
    torch.cuda.synchronize()
    _barrier(ws)
    clocks = clk.stop()
    ms = _max_over_ranks(e0.elapsed_time(e1), ws, dev) / (reps * TREE_REPLAYS)
    # the rows each launch read: the same calls again, untimed (same coins)
    rows_read = 0
    acc = np.zeros(N, np.int64)
    st_bad = 0
    for r in range(reps):
        o = ss.spec_verify_tree(pool[r % 2], *trees[r % 2], temperature=T, seed=11, step=r, workspace=wsv,
                                out=res)
        L = o["accept_len"].cpu().numpy()
        st_bad += int((o["status"].cpu().numpy() != 0).sum())
        rows_read += int((L + 1).sum())
        acc += np.bincount(L, minlength=N)[:N]
    alg = rows_read / reps * V * 2
    ach = alg / (ms / 1e3) / 1e9
    cpu = None
    if rank == 0:
        # the oracle on a sample: 32 sequences of both step tensors, 2 steps each
        nb = 32
        host = [p[:nb].float().cpu().numpy() for p in pool]
        htree = [tuple(a[:nb].cpu().numpy() for a in t) for t in trees]
        t0 = time.perf_counter()
        agree = 0
        for r in range(4):
            ob = oracle.tree_verify(host[r % 2], *htree[r % 2], temperature=T, seed=11, step=r)
            gb = ss.spec_verify_tree(pool[r % 2], *trees[r % 2], temperature=T, seed=11, step=r,
                                     workspace=wsv, out=res)
            agree += int((gb["accept_len"][:nb].cpu().numpy() == ob["accept_len"]).sum())
        el = time.perf_counter() - t0
        cpu = {"value": round(4 * nb / el, 2), "unit": "seq-steps/s", "cores": 1, "kind": "oracle",
               "sample": f"{nb} sequences x 4 steps of the same trees and coins ({el:.2f} s, fp64); "
                         f"{agree}/{4 * nb} accepted depths equal to the device's"}
    line = {"metric": "tree-draft verification seq-steps/s", "value": round(B / (ms / 1e3), 1),
            "unit": "seq-steps/s", "n_gpus": ws, "steps": reps, "warmup": max(args.warmup, 3),
            "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "tree_b256", "B": B, "N": N, "V": V, "temperature": T,
                       "tree_parent": list(TREE_PARENT), "l2": "two 622 MB step tensors alternate",
                       "timing": f"CUDA graph of {reps} verify launches, replayed {TREE_REPLAYS} times"},
            "roofline": {"bound": "hbm", "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s",
                         "frac": round(ach / hbm, 4), "traffic": _verify_traffic("tree_b256"),
                         "peak_source": peak_kind, "algorithmic_bytes_per_launch": round(alg, 1)},
            "cpu_baseline": cpu, "gpu_launches": reps * TREE_REPLAYS, "clocks": clocks,
            "breakdown": {"mean_accept": round(float((acc * np.arange(N)).sum() / acc.sum()), 4),
                          "accept_hist": acc.tolist(), "rows_per_seq": round(rows_read / reps / B, 4),
                          "bad_status": st_bad}}
    if rank == 0:
        print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------
# per-request sampling parameters
# --------------------------------------------------------------------------

SAMPLING_T = (0.6, 0.8, 1.0)
SAMPLING_TOP_K = (0, 20, 50)
SAMPLING_TOP_P = (0.9, 0.95, 1.0)


def run_sampling(args, ws, rank, dev):
    """B=256 sequences, K=3 one-hot drafts (uniform among each row's top 5),
    V=151936, bf16 logits N(0, sd 2); per sequence a temperature from
    {0.6, 0.8, 1.0}, top_k from {off, 20, 50} and top_p from {0.9, 0.95, 1.0}
    (seeded).  One step = spec_verify_sampling: the cut of all 4 rows of every
    sequence, then the verification with the cuts.  Two step tensors of 311 MB
    alternate (each above L2); CUDA graphs of the steps, and of the cut alone
    for its share."""
    import torch

    import oracle
    import sam_drafting_verification_gb300 as ss
    B, K, V = 256, 3, workloads.V_LARGE
    reps = min(max(args.steps, 1), 1000)
    hbm, peak_kind = _peaks()
    rng = np.random.default_rng(1008 + 7919 * rank)
    T = torch.tensor(rng.choice(SAMPLING_T, B), dtype=torch.float32, device=dev)
    k = torch.tensor(rng.choice(SAMPLING_TOP_K, B), dtype=torch.int32, device=dev)
    p = torch.tensor(rng.choice(SAMPLING_TOP_P, B), dtype=torch.float32, device=dev)
    pool = [workloads.sweep_device(9000 + i + 100 * rank, B, K, V, torch.bfloat16, dev) for i in range(2)]
    wsv = ss.verify_workspace(B, K, V, dev, sampling=True)
    res = ss.spec_verify_sampling(pool[0][0], pool[0][1], None, T, k, p, seed=3, step=0, workspace=wsv)
    tau = ss.sampling_cut(pool[0][0], T, k, p)
    for w in range(max(args.warmup, 3)):
        ss.spec_verify_sampling(pool[w % 2][0], pool[w % 2][1], None, T, k, p, seed=3, step=w,
                                workspace=wsv, out=res)
    torch.cuda.synchronize()
    cs = torch.cuda.Stream(device=dev)

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        cs.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(cs):
            with torch.cuda.graph(g, stream=cs):
                for r in range(reps):
                    fn(r)
        torch.cuda.synchronize()
        return g

    g_all = capture(lambda r: ss.spec_verify_sampling(pool[r % 2][0], pool[r % 2][1], None, T, k, p, seed=3,
                                                      step=r, workspace=wsv, out=res))
    lib = ss._b.lib()
    tau_ptr = tau.data_ptr()

    def cut_only(r):
        lg = pool[r % 2][0]
        ss._b.check(lib.spec_sampling_cut(lg.data_ptr(), ss.BF16, B, K + 1, V, T.data_ptr(), k.data_ptr(),
                                          p.data_ptr(), tau_ptr, cs.cuda_stream), "spec_sampling_cut")

    g_cut = capture(cut_only)

    def timed(g):
        _barrier(ws)
        torch.cuda.synchronize()
        with torch.cuda.stream(cs):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(cs)
            g.replay()
            e1.record(cs)
        torch.cuda.synchronize()
        _barrier(ws)
        return _max_over_ranks(e0.elapsed_time(e1), ws, dev) / reps

    clk = ClockSampler(dev.index or 0)
    clk.start()
    ms = timed(g_all)
    clocks = clk.stop()
    ms_cut = timed(g_cut)
    # rows the verification read: the same calls again, untimed
    rows_read = 0
    for r in range(min(reps, 200)):
        o = ss.spec_verify_sampling(pool[r % 2][0], pool[r % 2][1], None, T, k, p, seed=3, step=r,
                                    workspace=wsv, out=res)
        rows_read += int((o["accept_len"].cpu().numpy() + 1).sum())
        assert (o["status"] == 0).all()
    rows_per_seq = rows_read / min(reps, 200) / B
    # cut: once from HBM every row that has a truncation (no top-k and top_p
    # >= 1 leave a row unread); verification: the rows its chains needed
    kh_all, ph_all = k.cpu().numpy(), p.cpu().numpy()
    cut_seqs = int((((kh_all > 0) & (kh_all < V)) | (ph_all < 1.0)).sum())
    alg_cut = cut_seqs * (K + 1) * V * 2
    alg_ver = rows_per_seq * B * V * 2
    ach = alg_cut / (ms_cut / 1e3) / 1e9  # the cut kernel: each truncated row read once
    cpu = None
    if rank == 0:
        nb = 16
        host = [(pl[0][:nb].float().cpu().numpy(), pl[1][:nb].cpu().numpy()) for pl in pool]
        Th, kh, ph = (x[:nb].cpu().numpy() for x in (T, k, p))
        t0 = time.perf_counter()
        nst = 0  # steps over the two pools until about 10 s of host work
        while nst < 2 or (time.perf_counter() - t0 < 10.0 and nst < 1000):
            oracle.verify_sampling(host[nst % 2][0], host[nst % 2][1], None, Th, kh, ph, seed=3, step=nst)
            nst += 1
        el = time.perf_counter() - t0
        cpu = {"value": round(nst * nb / el, 2), "unit": "seq-steps/s", "cores": 1, "kind": "oracle",
               "sample": f"{nb} sequences x {nst} steps over two pools of logits, the same parameters "
                         f"({el:.2f} s, fp64)"}
    line = {"metric": "sampling-parameter verification seq-steps/s", "value": round(B / (ms / 1e3), 1),
            "unit": "seq-steps/s", "n_gpus": ws, "steps": reps, "warmup": max(args.warmup, 3),
            "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "sampling_b256", "B": B, "K": K, "V": V,
                       "temperature": list(SAMPLING_T), "top_k": list(SAMPLING_TOP_K),
                       "top_p": list(SAMPLING_TOP_P), "l2": "two 311 MB step tensors alternate",
                       "timing": f"CUDA graph of {reps} steps (cut + verify launches)"},
            "roofline": {"kernel": "cut_hist_kernel (bf16)", "bound": "hbm", "achieved": round(ach, 1), "peak": hbm,
                         "unit": "GB/s", "frac": round(ach / hbm, 4),
                         "traffic": _traffic(CUT_TRAFFIC, "sampling_b256", "sampling.cu"),
                         "peak_source": peak_kind, "algorithmic_bytes_per_launch": round(alg_cut, 1),
                         "algorithmic_bytes_per_step": round(alg_cut + alg_ver, 1)},
            "cpu_baseline": cpu, "gpu_launches": 3 * reps, "clocks": clocks,
            "breakdown": {"cut_us": round(ms_cut * 1e3, 2), "verify_us": round((ms - ms_cut) * 1e3, 2),
                          "cut_GBps_one_read": round(alg_cut / (ms_cut / 1e3) / 1e9, 1),
                          "rows_per_seq": round(rows_per_seq, 4)}}
    if rank == 0:
        print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------
# reference arm: the oracle
# --------------------------------------------------------------------------

REF_SEQS = 16


def run_reference(args):
    """The oracle arm on the default line's workload: one step = the oracle's
    fp64 verification of 16 sequences of B=1024, K=3, bf16, T=1 inputs (same
    distributions, drawn on the host), single-threaded."""
    import oracle
    ws, rank, local = _dist()
    if rank != 0:
        return
    rows, drafts = workloads.sweep_host_bf16(HEAD_SEED, REF_SEQS, HEAD_K)
    si = np.arange(REF_SEQS)
    for s in range(max(args.warmup, 0)):
        oracle.verify(rows, drafts, None, temperature=HEAD_T, seed=HEAD_COIN_SEED, step=s, seq_index=si)
    t0 = time.perf_counter()
    for s in range(args.steps):
        oracle.verify(rows, drafts, None, temperature=HEAD_T, seed=HEAD_COIN_SEED, step=1000 + s, seq_index=si)
    el = time.perf_counter() - t0
    v = REF_SEQS * args.steps / el if el > 0 else 0.0
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 2), "unit": "seq-steps/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(el / max(args.steps, 1) * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": head_config(1),
            "cpu_baseline": {"value": round(v, 2), "unit": "seq-steps/s", "cores": 1, "kind": "oracle",
                             "nproc": _nproc(),
                             "sample": f"each step: fp64 verification of {REF_SEQS} sequences of the "
                                       f"workload (host-drawn, same distributions), one thread"},
            "e2e": {"value": round(v, 2), "unit": "seq-steps/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_gpu(args):
    import torch

    import sam_drafting_verification_gb300  # noqa: F401  (fails loudly without the library)
    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)
    run = {"verify_b1024": run_verify_b1024, "rs_bf16_b64": run_rs, "sweep_b1024": run_sweep,
           "long_rollout_b256": run_rollout, "draft_model_b32": run_draft_model,
           "rollout_toy_b64": run_rollout_toy, "static_match_b256": run_static_match,
           "tree_b256": run_tree, "sampling_b256": run_sampling}[args.workload]
    run(args, ws, rank, dev)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


WORKLOADS = ["verify_b1024", "rs_bf16_b64", "sweep_b1024", "long_rollout_b256", "draft_model_b32",
             "rollout_toy_b64", "static_match_b256", "tree_b256", "sampling_b256"]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="verify_b1024", choices=WORKLOADS)
    ap.add_argument("--point", default="", help="sweep_b1024 only: one point 'K,f32|bf16,greedy|T=1|greedy-full-read'")
    ap.add_argument("--pool", type=int, default=HEAD_POOL,
                    help="verify_b1024 only: logits tensors the steps rotate through")
    ap.add_argument("--no-breakdown", action="store_true",
                    help="verify_b1024 only: the default line without the other configurations")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "gb300":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
