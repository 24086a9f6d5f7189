"""Benchmark of the SAM-drafting + lossless-verification hot path on GB300.

One step = one pass of the per-step hot path over a batch: the device suffix
automata are extended with the tokens the previous verification emitted and
queried for K drafts (sam_step, one launch), then the drafts are verified
against that step's target logits (spec_verify, one launch).  The emitted
tokens feed the next step, as in a decode loop.

Default workload (rs_bf16_b64): B=64 sequences per GPU, V=151936, Zipf(1.1)
histories of 4096 tokens (copy prob 0.3, spans 8-64), K=3 SAM drafts,
rejection sampling at T=1.0 on bf16 logits N(0, sd 2) + 4 on the stream's
true continuation.  Logits come from a rotating pool of 16 step tensors
(1.24 GB, far above the 129 MB L2), so no step finds its rows in L2.

The timed region replays a CUDA graph of exactly --steps steps, bracketed by a
barrier and a device synchronisation, timed with CUDA events on the capture
stream; max over ranks.  Under torchrun every rank runs its own batch (weak
scaling, no collective on the data path).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                  [--workload rs_bf16_b64|sweep_b1024|long_rollout_b256|rollout_toy_b64|static_match_b256|tree_b256|sampling_b256]
"""
from __future__ import annotations

import argparse
import json
import os
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

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per launch of the
# verify kernel, from the ncu captures summarised under profiles/, keyed by
# workload, with the SHA-256 of verify.cu they were taken on: a changed kernel
# reports null until it is captured again.
VERIFY_TRAFFIC = {
    "rs_bf16_b64": {"bytes": 19537920.0, "profile": "profiles/verify_kernel_rs_bf16_b64.md",
                    "verify_cu_sha256": "bbb652d498d8e15843e7c24655bb1eb7a46a9b7e25e1c39905f50390e090f3fe"},
    "long_rollout_b256": {"bytes": 78981542.0, "profile": "profiles/launches_long_rollout_b256.md",
                          "verify_cu_sha256": "501dfc92dfa938d5aaadc35a389107c2249f8a4a90a8c3e282f45d804219eb47"},
    "tree_b256": {"bytes": 161624064.0, "profile": "profiles/verify_kernel_tree_b256.md",
                  "verify_cu_sha256": "501dfc92dfa938d5aaadc35a389107c2249f8a4a90a8c3e282f45d804219eb47"},
}
# the same for the sampling cut kernel (sampling.cu)
CUT_TRAFFIC = {"sampling_b256": {"bytes": 277559040.0, "profile": "profiles/cut_hist_kernel_sampling_b256.md",
                                 "sampling_cu_sha256": "78f29c9034b75bbbe1bded1e886e3e513b3184c3ee3411e7902190e5669d7d55"}}


def _traffic(table, workload, source):
    import hashlib
    t = table.get(workload)
    if t is None:
        return None
    src = os.path.join(ROOT, "sam_drafting_verification_gb300", "csrc", source)
    with open(src, "rb") as f:
        if hashlib.sha256(f.read()).hexdigest() != t[source.replace(".", "_") + "_sha256"]:
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
# inputs of the default workload
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


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------

def run_gpu(args):
    import torch

    import sam_drafting_verification_gb300 as ss

    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)
    if args.workload == "sweep_b1024":
        return run_sweep(args, ws, rank, dev)
    if args.workload == "long_rollout_b256":
        return run_rollout(args, ws, rank, dev)
    if args.workload == "rollout_toy_b64":
        return run_rollout_toy(args, ws, rank, dev)
    if args.workload == "static_match_b256":
        return run_static_match(args, ws, rank, dev)
    if args.workload == "tree_b256":
        return run_tree(args, ws, rank, dev)
    if args.workload == "sampling_b256":
        return run_sampling(args, ws, rank, dev)

    B, V, K, T, n = 64, workloads.V_LARGE, 3, 1.0, 4096
    hist, cont = rs_inputs(rank, B, V, n, K)
    steps, warm = args.steps, args.warmup
    cap = n + (K + 1) * (steps + warm + 8) + 64
    batch = ss.SamBatch(B, cap, V, device=dev)
    hist_d = torch.as_tensor(hist, device=dev)
    nfull = torch.full((B,), n, dtype=torch.int32, device=dev)

    # S1: prefill build (one launch), timed on its own
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
    draft = torch.empty((B, K), dtype=torch.int32, device=dev)
    dlen = torch.empty(B, dtype=torch.int32, device=dev)
    mlen = torch.empty(B, dtype=torch.int32, device=dev)
    mend = torch.empty(B, dtype=torch.int32, device=dev)
    out = {"accept_len": torch.empty(B, dtype=torch.int32, device=dev),
           "out_token": torch.empty(B, dtype=torch.int32, device=dev),
           "emit": emit, "emit_len": emit_len,
           "status": torch.empty(B, dtype=torch.int32, device=dev)}
    acc_log = torch.zeros((max(min(steps, 2000), 1), B), dtype=torch.int32, device=dev)
    wsv = ss.verify_workspace(B, K, V, dev)

    def step(s, log_row=None, only_verify=False):
        if not only_verify:
            batch.step(emit, emit_len, K, out=(draft, dlen, mlen, mend))
        ss.spec_verify(pool[s % POOL], draft, dlen, temperature=T, seed=1002, step=s, out=out,
                       emit=True, status=True, workspace=wsv)
        if log_row is not None:
            log_row.copy_(out["accept_len"])

    # warm-up (eager), then restore the automata to the post-prefill snapshot
    for s in range(warm):
        step(s)
    torch.cuda.synchronize()
    batch.import_(snap)
    emit_len.zero_()

    # capture exactly `steps` steps (2 kernels each) in one graph
    cs = torch.cuda.Stream(device=dev)
    g = torch.cuda.CUDAGraph()
    cs.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(cs):
        with torch.cuda.graph(g, stream=cs):
            for s in range(steps):
                step(warm + s)
    torch.cuda.synchronize()
    batch.import_(snap)
    emit_len.zero_()
    torch.cuda.synchronize()

    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)
    _barrier(ws)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.nvtx.range_push("timed")
    t0.record()
    g.replay()
    t1.record()
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    _barrier(ws)
    total_ms = t0.elapsed_time(t1)
    clk = clocks.stop()
    st = out["status"].cpu().numpy()
    assert (st == 0).all() and (batch.status() == 0).all(), "verification or automaton error"

    # acceptance of the first timed steps (eager re-run of the same steps, outside timing)
    n_acc = min(steps, 2000)
    batch.import_(snap)
    emit_len.zero_()
    for s in range(n_acc):
        step(warm + s, log_row=acc_log[s])
    torch.cuda.synchronize()
    L = acc_log[:n_acc].cpu().numpy().astype(np.int64)

    # attribution: the verify launches alone, replayed as a graph on the same inputs
    n_att = min(steps, 2000)
    gv = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cs):
        with torch.cuda.graph(gv, stream=cs):
            for s in range(n_att):
                step(warm + s, only_verify=True)
    torch.cuda.synchronize()
    v0, v1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    v0.record()
    gv.replay()
    v1.record()
    torch.cuda.synchronize()
    verify_ms = v0.elapsed_time(v1) / n_att
    Lv = out["accept_len"].cpu().numpy().astype(np.int64)  # last verify's lengths (same drafts each launch)

    ms_step = _max_over_ranks(total_ms / steps, ws, dev)
    seqs = _sum_over_ranks(float(B), ws, dev)
    value = seqs / (ms_step / 1e3)
    sam_ms = max(ms_step - verify_ms, 0.0)

    # verify roofline: algorithmic bytes = rows the accept chains need
    row_bytes = V * 2
    verify_bytes = float((Lv + 1).sum()) * row_bytes
    hbm, peak_kind = _peaks()
    achieved = verify_bytes / (verify_ms / 1e3) / 1e9
    roof = {"kernel": "verify_kernel<bf16, one-hot, T>0>", "bound": "hbm",
            "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
            "frac": round(achieved / hbm, 4), "traffic": _verify_traffic("rs_bf16_b64"),
            "peak_source": f"{peak_kind} hbm_gbs (burst copy)",
            "algorithmic_bytes_per_launch": verify_bytes,
            "kernel_ms": round(verify_ms, 5)}

    cpu = cpu_baseline_rs(hist, cont) if rank == 0 else None
    e2e = e2e_rs(batch, snap, pool, emit, emit_len, draft, dlen, mlen, mend, out, wsv, B, K, V, T,
                 steps=min(steps, 200), dev=dev)

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "seq-steps/s", "n_gpus": ws,
        "steps": steps, "warmup": warm, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32 (bf16 logits)", "data": "synthetic",
        "config": {"workload": "rs_bf16_b64", "B_per_gpu": B, "V": V, "K": K, "temperature": T,
                   "history": n, "logits": "bf16 N(0, sd 2) + 4 on the true continuation",
                   "drafts": "device SAM (K=3)", "parallelism": f"dp{ws} (independent batches)",
                   "l2": f"inputs larger than L2: rotating pool of {POOL} logits tensors "
                         f"({POOL * B * (K + 1) * V * 2 / 1e9:.2f} GB)",
                   "timing": "CUDA graph of exactly `steps` steps, events on the capture stream"},
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": 2 * steps,
        "clocks": clk,
        "breakdown": {
            "sam_step_ns_per_seq_step": round(sam_ms * 1e6 / B, 1),
            "verify_us_per_step": round(verify_ms * 1e3, 2),
            "verify_algorithmic_GBps": round(achieved, 1),
            "prefill_tokens_per_s": round(B * n / (prefill_ms / 1e3), 1),
            "mean_accept_len": round(float(L.mean()), 4),
            "mean_emitted_per_step": round(float(L.mean()) + 1, 4),
        },
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def e2e_rs(batch, snap, pool, emit, emit_len, draft, dlen, mlen, mend, out, wsv, B, K, V, T, steps, dev):
    """Same metric through the public API with host buffers: every step copies
    its logits from pinned host memory and reads the emitted tokens back.  The
    copy of step s + 1 runs on a copy stream into a second device buffer while
    step s computes (the host link, about 200 GB/s, bounds the loop)."""
    import torch

    import sam_drafting_verification_gb300 as ss
    host_pool = [p.cpu().pin_memory() for p in pool[:4]]
    dev_buf = [torch.empty_like(pool[0]) for _ in range(2)]
    host_emit = torch.empty((B, K + 1), dtype=torch.int32).pin_memory()
    host_len = torch.empty(B, dtype=torch.int32).pin_memory()
    batch.import_(snap)
    emit_len.zero_()
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
            dev_buf[i].copy_(host_pool[s % len(host_pool)], non_blocking=True)
        copied[i].record(cps)

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(cur)
    cps.wait_stream(cur)
    issue_copy(0)
    for s in range(steps):
        if s + 1 < steps:
            issue_copy(s + 1)
        cur.wait_event(copied[s % 2])
        batch.step(emit, emit_len, K, out=(draft, dlen, mlen, mend))
        ss.spec_verify(dev_buf[s % 2], draft, dlen, temperature=T, seed=1002, step=s, out=out,
                       emit=True, status=True, workspace=wsv)
        freed[s % 2].record(cur)
        host_emit.copy_(emit, non_blocking=True)
        host_len.copy_(emit_len, non_blocking=True)
    e1.record(cur)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    return {"value": round(B / (ms / 1e3), 1), "unit": "seq-steps/s",
            "h2d_bytes_per_step": int(dev_buf[0].numel() * dev_buf[0].element_size()),
            "d2h_bytes_per_step": int(host_emit.numel() * 4 + host_len.numel() * 4),
            "ms_per_step": round(ms, 4), "steps": steps,
            "overlap": "step s + 1's copy on a second stream while step s computes"}


class OracleLoop:
    """The oracle as it stands, on a sample of the same workload: each sampled
    sequence's automaton is built over its history (untimed); a step extends it
    with the previously emitted tokens, drafts K and verifies the draft in fp64
    against that step's logits (host-generated, same distribution, bf16-rounded)."""

    def __init__(self, hist, cont, nseq, npool=4, seed=77):
        import torch

        import oracle
        self.oracle = oracle
        V, K = workloads.V_LARGE, 3
        self.K, self.T, self.nseq, self.npool = K, 1.0, nseq, npool
        rng = np.random.default_rng(seed)
        self.rows = []
        for p in range(npool):
            x = workloads.gaussian_logits(rng, (nseq, K + 1, V), 2.0)
            workloads.boost_truth(x, cont[:nseq, p * (K + 1):(p + 1) * (K + 1)], 4.0)
            self.rows.append(workloads.to_bf16(x).float().numpy())
        self.sams = [oracle.Sam(V) for _ in range(nseq)]
        for b in range(nseq):
            self.sams[b].extend(hist[b])
        self.emit = [[] for _ in range(nseq)]

    def seq_step(self, b, s):
        K = self.K
        self.sams[b].extend(self.emit[b])
        d, dl, _, _ = self.sams[b].draft(K)
        d = np.maximum(d, 0)[None]
        rows = self.rows[s % self.npool][b:b + 1]
        r = self.oracle.verify(rows, d, np.array([dl], np.int32), temperature=self.T, seed=1002,
                               step=s, seq_index=np.array([b]))
        L = int(r["accept_len"][0])
        self.emit[b] = list(d[0, :L]) + [int(r["out_token"][0])]


def cpu_baseline_rs(hist, cont, nseq=64, min_steps=40, target_s=10.0, max_steps=1000):
    """The oracle's decode steps over nseq sequences, repeated until about
    target_s seconds of host work (at least min_steps steps)."""
    loop = OracleLoop(hist, cont, nseq)
    t0 = time.perf_counter()
    nsteps = 0
    while nsteps < max_steps and (nsteps < min_steps or time.perf_counter() - t0 < target_s):
        for b in range(nseq):
            loop.seq_step(b, nsteps)
        nsteps += 1
    el = time.perf_counter() - t0
    return {"value": round(nseq * nsteps / el, 2), "unit": "seq-steps/s", "cores": 1, "kind": "oracle",
            "sample": f"{nseq} sequences x {nsteps} decode steps of the same workload "
                      f"(extend + draft + fp64 verify, single thread), {el:.2f} s"}


# --------------------------------------------------------------------------
# long-tail rollout: B=256 long histories, 512 decode steps
# --------------------------------------------------------------------------

def run_rollout(args, ws, rank, dev):
    """B=256 histories log-uniform in [16k, 32k] tokens (Zipf(1.1), copy prob
    0.5, spans 16-256), V=151936: one prefill build, then 512 steps of
    (extend by the stream's next U{1..4} tokens + draft K=3, greedy verify of
    the drafts on bf16 logits [256, 4, V] ~ N(0, sd 2)).  The SAM step is also
    timed alone (ns per sequence-step) next to the oracle's extend + draft on
    a sample of the same sequences."""
    import torch

    import sam_drafting_verification_gb300 as ss
    w = workloads.long_rollout(seed=1004 + 7919 * rank)
    B, V, K, steps = w["B"], w["V"], w["K"], w["steps"]
    lens, n_new, streams = w["lens"], w["n_new"], w["streams"]
    cap = int(max(len(x) for x in streams))
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
    batch = ss.SamBatch(B, cap, V, device=dev)
    pre_d = torch.as_tensor(pre, device=dev)
    lens_d = torch.as_tensor(lens, device=dev)
    toks_d = torch.as_tensor(toks, device=dev)
    nn_d = torch.as_tensor(n_new, device=dev)

    # S1: prefill (one launch), timed after one untimed build
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

    npool = 4  # 4 x 311 MB of bf16 logits: each step's rows are not in L2
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

    def step(s, sam=True, verify=True):
        if sam:
            batch.step(toks_d[s], nn_d[s], K, out=(draft, dlen, mlen, mend))
        if verify:
            ss.spec_verify(pool[s % npool], draft, dlen, temperature=0.0, out=out, status=True,
                           workspace=wsv)

    def graph(**kw):
        cs = torch.cuda.Stream(device=dev)
        gr = torch.cuda.CUDAGraph()
        cs.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(cs):
            with torch.cuda.graph(gr, stream=cs):
                for s in range(steps):
                    step(s, **kw)
        torch.cuda.synchronize()
        return gr

    def timed(gr):
        batch.import_(snap)
        torch.cuda.synchronize()
        _barrier(ws)
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        gr.replay()
        b_.record()
        torch.cuda.synchronize()
        _barrier(ws)
        return a.elapsed_time(b_)

    for s in range(max(args.warmup, 3)):  # eager warm-up
        step(s)
    torch.cuda.synchronize()
    batch.import_(snap)
    g_full = graph()
    g_sam = graph(verify=False)
    timed(g_full)  # graph warm-up
    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)
    full_ms = timed(g_full)
    clk = clocks.stop()
    assert (out["status"].cpu() == 0).all() and (batch.status() == 0).all()
    sam_ms = timed(g_sam)
    # drafts of the last step: the automata followed the streams exactly
    st_ms = _max_over_ranks(full_ms / steps, ws, dev)
    sam_ns = _max_over_ranks(sam_ms / steps / B * 1e6, ws, dev)
    seqs = _sum_over_ranks(float(B), ws, dev)
    verify_ms = max(full_ms - sam_ms, 1e-9) / steps
    Lh = out["accept_len"].cpu().numpy().astype(np.int64)
    hbm, peak_kind = _peaks()
    vbytes = float((Lh + 1).sum()) * V * 2
    achieved = vbytes / (verify_ms / 1e3) / 1e9

    cpu = None
    if rank == 0:
        cpu = oracle_sam_rollout(streams, lens, toks, n_new, K, nseq=B)
    line = {
        "metric": METRIC, "value": round(seqs / (st_ms / 1e3), 1), "unit": "seq-steps/s",
        "n_gpus": ws, "steps": steps, "warmup": max(args.warmup, 3), "ms_per_step": round(st_ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32 (SAM), f32 (bf16 logits)",
        "data": "synthetic",
        "config": {"workload": "long_rollout_b256", "B_per_gpu": B, "V": V, "K": K, "steps": steps,
                   "history": "log-uniform [16384, 32768]", "prefill_tokens": int(lens.sum()),
                   "verify": "greedy, bf16 N(0, sd 2)",
                   "l2": f"inputs larger than L2: {npool} logits tensors of {B * (K + 1) * V * 2 / 1e6:.0f} MB",
                   "timing": "CUDA graph of the 512 steps, events on the capture stream"},
        "roofline": {"kernel": "verify_kernel<bf16, greedy>", "bound": "hbm", "achieved": round(achieved, 1),
                     "peak": hbm, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                     "traffic": _verify_traffic("long_rollout_b256"),
                     "peak_source": f"{peak_kind} hbm_gbs (burst copy)",
                     "algorithmic_bytes_per_launch": vbytes,
                     "note": "verify time = (full step - SAM-only step) / steps"},
        "cpu_baseline": cpu,
        "gpu_launches": 2 * steps,
        "clocks": clk,
        "breakdown": {
            "sam_step_ns_per_seq_step": round(sam_ns, 1),
            "sam_vs_oracle": (round(cpu["value"] / sam_ns, 1) if cpu else None),
            "verify_us_per_step": round(verify_ms * 1e3, 2),
            "prefill_tokens_per_s": round(float(lens.sum()) / (prefill_ms / 1e3), 1),
            "prefill_ms": round(prefill_ms, 3),
        },
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def oracle_sam_rollout(streams, lens, toks, n_new, K, nseq):
    """The oracle's extend + draft (one C call per step for the sample), on
    the first nseq sequences of the rollout; the builds are untimed."""
    import oracle
    V = workloads.V_LARGE
    sams = [oracle.Sam(V) for _ in range(nseq)]
    for b in range(nseq):
        sams[b].extend(streams[b][:lens[b]])
    steps = toks.shape[0]
    t0 = time.perf_counter()
    for s in range(steps):
        oracle.step_batch(sams, toks[s, :nseq], n_new[s, :nseq], K)
    el = time.perf_counter() - t0
    return {"value": round(el / (steps * nseq) * 1e9, 1), "unit": "ns/seq-step (SAM extend + draft)",
            "cores": 1, "kind": "oracle",
            "sample": f"{nseq} of the 256 sequences x {steps} steps, single thread, {el:.2f} s"}


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
# verification sweep at B=1024
# --------------------------------------------------------------------------

def run_sweep(args, ws, rank, dev):
    import torch

    import sam_drafting_verification_gb300 as ss
    B, V = 1024, workloads.V_LARGE
    hbm, peak_kind = _peaks()
    points = []
    reps = max(args.steps, 1)
    only = None
    if args.point:  # "K,dtype,mode", e.g. "3,bf16,T=1": one sweep point (profiling)
        k_s, d_s, m_s = args.point.split(",")
        only = (int(k_s), {"f32": torch.float32, "bf16": torch.bfloat16}[d_s], m_s)
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
                for _ in range(args.warmup):
                    ss.spec_verify(logits, dr, None, temperature=T, seed=5, step=0, out=res, workspace=wsv)
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                for r in range(reps):
                    ss.spec_verify(logits, dr, None, temperature=T, seed=5, step=r, out=res, workspace=wsv)
                e1.record()
                torch.cuda.synchronize()
                ms = e0.elapsed_time(e1) / reps
                Lh = res["accept_len"].cpu().numpy().astype(np.int64)
                alg = float((Lh + 1).sum()) * V * logits.element_size()
                points.append({"K": K, "dtype": str(dtype).split(".")[-1], "mode": name,
                               "us": round(ms * 1e3, 2), "seq_steps_per_s": round(B / (ms / 1e3), 1),
                               "mean_accept": round(float(Lh.mean()), 4),
                               "alg_GBps": round(alg / (ms / 1e3) / 1e9, 1),
                               "frac": round(alg / (ms / 1e3) / 1e9 / hbm, 4)})
            del logits, draft, full_draft
            torch.cuda.empty_cache()
    head = max(points, key=lambda p: p["frac"])
    line = {"metric": METRIC, "value": head["seq_steps_per_s"], "unit": "seq-steps/s", "n_gpus": ws,
            "steps": reps, "warmup": args.warmup, "ms_per_step": head["us"] / 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": {"workload": "sweep_b1024", "B": B, "V": V},
            "roofline": {"bound": "hbm", "achieved": head["alg_GBps"], "peak": hbm, "unit": "GB/s",
                         "frac": head["frac"], "traffic": None, "peak_source": peak_kind},
            "points": points}
    if rank == 0:
        print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------
# reference arm: the oracle
# --------------------------------------------------------------------------

def run_reference(args):
    """The oracle arm: one step = one sequence's decode step (extend + draft +
    fp64 verification) of the same workload, single-threaded on the host."""
    ws, rank, local = _dist()
    if rank != 0:
        return
    hist, cont = rs_inputs(0)
    nseq = 8
    loop = OracleLoop(hist, cont, nseq)
    for s in range(max(args.warmup, 0)):
        loop.seq_step(s % nseq, s // nseq)
    t0 = time.perf_counter()
    for s in range(args.steps):
        loop.seq_step(s % nseq, 1000 + s // nseq)
    el = time.perf_counter() - t0
    v = args.steps / el if el > 0 else 0.0
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 2), "unit": "seq-steps/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 / v, 3) if v else None, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "rs_bf16_b64", "B_per_gpu": 64, "V": workloads.V_LARGE, "K": 3,
                       "temperature": 1.0, "history": 4096},
            "cpu_baseline": {"value": round(v, 2), "unit": "seq-steps/s", "cores": 1, "kind": "oracle",
                             "sample": f"each step: one sequence's decode step, {nseq} sequences in turn"},
            "e2e": {"value": round(v, 2), "unit": "seq-steps/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="rs_bf16_b64", choices=["rs_bf16_b64", "sweep_b1024", "long_rollout_b256",
                                                      "rollout_toy_b64", "static_match_b256", "tree_b256",
                                                      "sampling_b256"])
    ap.add_argument("--point", default="", help="sweep_b1024 only: one point 'K,f32|bf16,greedy|T=1|greedy-full-read'")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "gb300":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
