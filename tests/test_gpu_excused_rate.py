"""Excused decisions at the benchmark vocabulary, counted over a large fixed
sample: V=151936, B=256, one draft per sequence (among its row's top 5),
logits N(0, sd 2), fp32 and bf16, T in {0.7, 1, 2}, 36 coin draws (steps)
each -- about 111k accept/resample decisions.

A GPU decision may differ from the oracle's only where its uniform lies within
1e-6 of the oracle's threshold or CDF boundary (checked per decision by
compare_verify), and such decisions must stay at or below 1e-4 of all
decisions.  Inputs and coins are seeded and the kernel is deterministic, so
the count is reproducible.  The oracle runs in a pool of spawned processes."""
import multiprocessing as mp
import os

import numpy as np
import pytest
import torch

import workloads
from parity import compare_verify, gpu_to_numpy

pytestmark = pytest.mark.gpu

B, K, V, STEPS = 256, 1, 151936, 36


def _oracle_call(args):
    import oracle
    rows, draft, T, step = args
    return oracle.verify(rows, draft, None, temperature=T, seed=21, step=step)


def test_excused_rate_at_full_vocabulary(cuda_device):
    import sam_drafting_verification_gb300 as ss
    ctx = mp.get_context("spawn")
    decisions = excused = 0
    with ctx.Pool(max(2, min(16, (os.cpu_count() or 4) - 1))) as pool:
        for T in (1.0, 0.7, 2.0):
            for dtype in (torch.float32, torch.bfloat16):
                logits, draft = workloads.sweep_host(4100 + int(T * 10), B, K, V)
                tt = torch.from_numpy(logits).to(dtype)
                rows = tt.float().numpy()
                dg = torch.as_tensor(draft, device=cuda_device)
                td = tt.to(cuda_device)
                gs = [gpu_to_numpy(ss.spec_verify(td, dg, None, temperature=T, seed=21, step=s, debug=True))
                      for s in range(STEPS)]
                outs = pool.map(_oracle_call, [(rows, draft, T, s) for s in range(STEPS)])
                for g, o in zip(gs, outs):
                    d, e = compare_verify(g, o, lambda b: rows[b], draft, None, T, check_probs=False,
                                          budget=False)
                    decisions += d
                    excused += e
    assert decisions > 100000
    assert excused <= 1e-4 * decisions, f"{excused} excused of {decisions}"


# ---- per-request sampling parameters and draft trees --------------------------

SAMP_B, SAMP_STEPS, SAMP_SEEDS = 256, 52, (4301, 4302)
TREE_B, TREE_STEPS = 128, 72
TREE_PARENT = (-1, 0, 1, 2, 0, 4, 5, 0)
TREE_BOOST = (0.0, 14.0, 14.0, 14.0, 12.0, 12.0, 12.0, 11.0)
_cache = {}


def sampling_inputs(seed, bf16):
    """B=256, K=1, V=151936 rows N(0, sd 2) (bf16-rounded or not), the draft
    among its row's top 5, and per sequence T in {0.6, 0.8, 1}, top_k in
    {off, 20, 50, 1000}, top_p in {0.9, 0.95, 1}."""
    rng = np.random.default_rng(seed)
    logits = workloads.gaussian_logits(rng, (SAMP_B, 2, V), 2.0)
    if bf16:
        logits = workloads.round_bf16(logits)
    draft = workloads.topk_drafts(logits[:, :1], 5, rng)
    T = rng.choice([0.6, 0.8, 1.0], SAMP_B).astype(np.float32)
    k = rng.choice([0, 20, 50, 1000], SAMP_B).astype(np.int32)
    p = rng.choice([0.9, 0.95, 1.0], SAMP_B).astype(np.float32)
    return logits, draft, T, k, p


def tree_inputs(seed):
    """TREE_B trees of 8 nodes (three candidates under the root, two of them
    with chains of two more), V=151936, rows N(0, sd 2) with each node's
    token raised in its parent's row by 14 / 12 / 11 per branch."""
    rng = np.random.default_rng(seed)
    N = len(TREE_PARENT)
    logits = workloads.gaussian_logits(rng, (TREE_B, N, V), 2.0)
    fc = np.full(N, -1, np.int32)
    ns = np.full(N, -1, np.int32)
    last = {}
    for n in range(1, N):
        par = TREE_PARENT[n]
        if par in last:
            ns[last[par]] = n
        else:
            fc[par] = n
        last[par] = n
    tok = np.full((TREE_B, N), -1, np.int32)
    for b in range(TREE_B):
        t = rng.integers(0, V, N - 1)
        while len(set(t.tolist())) < N - 1:  # distinct tokens in a tree
            t = rng.integers(0, V, N - 1)
        tok[b, 1:] = t
        for n in range(1, N):
            logits[b, TREE_PARENT[n], tok[b, n]] += np.float32(TREE_BOOST[n])
    return logits, tok, np.tile(fc, (TREE_B, 1)), np.tile(ns, (TREE_B, 1))


def _oracle_sampling(args):
    import oracle
    seed, bf16, step = args
    key = ("s", seed, bf16)
    if key not in _cache:
        _cache.clear()
        _cache[key] = sampling_inputs(seed, bf16)
    logits, draft, T, k, p = _cache[key]
    return oracle.verify_sampling(logits, draft, None, T, k, p, seed=23, step=step)


def _oracle_tree(args):
    import oracle
    seed, T, step = args
    key = ("t", seed)
    if key not in _cache:
        _cache.clear()
        _cache[key] = tree_inputs(seed)
    logits, tok, fc, ns = _cache[key]
    return oracle.tree_verify(logits, tok, fc, ns, temperature=T, seed=29, step=step)


def test_excused_rate_sampling_parameters(cuda_device):
    """Verification under per-request temperature, top-k and top-p at
    V=151936 over about 100k decisions: every mismatch excused (a top-p cut
    within 1e-6 of its boundary in mass, or a coin within 1e-6 of its
    threshold or CDF boundary) and at most 1e-4 of the decisions."""
    import sam_drafting_verification_gb300 as ss
    from parity import compare_sampling
    ctx = mp.get_context("spawn")
    decisions = excused = 0
    with ctx.Pool(max(2, min(15, (os.cpu_count() or 4) - 1))) as pool:
        for seed in SAMP_SEEDS:
            for bf16 in (False, True):
                logits, draft, T, k, p = sampling_inputs(seed, bf16)
                dt = torch.bfloat16 if bf16 else torch.float32
                tl = torch.from_numpy(logits).to(dt).to(cuda_device)
                args = [torch.from_numpy(a).to(cuda_device) for a in (T, k, p)]
                dg = torch.as_tensor(draft, device=cuda_device)
                tau_g = ss.sampling_cut(tl, *args).cpu().numpy()
                gs = []
                for s in range(SAMP_STEPS):
                    g = ss.spec_verify_sampling(tl, dg, None, *args, seed=23, step=s)
                    gs.append({key: v.cpu().numpy() for key, v in g.items()})
                outs = pool.map(_oracle_sampling, [(seed, bf16, s) for s in range(SAMP_STEPS)], chunksize=3)
                for g, o in zip(gs, outs):
                    d, e = compare_sampling(g, o, logits, draft, T, k, p, tau_g, budget=False)
                    decisions += d
                    excused += e
    assert decisions > 100000
    assert excused <= 1e-4 * decisions, f"{excused} excused of {decisions}"


def test_excused_rate_trees(cuda_device):
    """Tree verification at V=151936 over about 100k decisions (T in {0.7, 1}):
    every mismatch excused (a depth's coin within 1e-6 of a child's running
    sum, or the final coin within 1e-6 of the oracle's interval of the GPU's
    token) and at most 1e-4 of the decisions."""
    import sam_drafting_verification_gb300 as ss
    from parity import compare_trees
    ctx = mp.get_context("spawn")
    decisions = excused = 0
    with ctx.Pool(max(2, min(8, (os.cpu_count() or 4) - 1))) as pool:
        for seed, T in ((4401, 1.0), (4402, 0.7), (4403, 1.0), (4404, 0.7)):
            logits, tok, fc, ns = tree_inputs(seed)
            tl = torch.from_numpy(logits).to(cuda_device)
            i32 = [torch.as_tensor(a, device=cuda_device) for a in (tok, fc, ns)]
            gs = []
            for s in range(TREE_STEPS):
                g = ss.spec_verify_tree(tl, *i32, temperature=T, seed=29, step=s)
                gs.append({key: v.cpu().numpy() for key, v in g.items()})
            outs = pool.map(_oracle_tree, [(seed, T, s) for s in range(TREE_STEPS)], chunksize=4)
            for s, (g, o) in enumerate(zip(gs, outs)):
                d, e = compare_trees(g, o, logits, tok, fc, ns, T, seed=29, step=s, budget=False)
                decisions += d
                excused += e
            del tl
    assert decisions > 100000
    assert excused <= 1e-4 * decisions, f"{excused} excused of {decisions}"
