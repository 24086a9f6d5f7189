"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke check.

This module only draws inputs.  It holds none of the method's arithmetic (no
automaton, softmax or verification): token streams with repeated spans, history
lengths, Gaussian logits with a boost on the stream's true continuation, and
draft tokens picked the way each workload prescribes.

Workloads (named by what they are):
  tiny          B=4, V=64, uniform-token streams of 256 with copied spans 4-16
                (prob 0.3), K=3, greedy, fp32 logits N(0,1) + 3 on the truth
  rs_bf16_b64   B=64, V=151936, Zipf(1.1) histories of 4096 (copy prob 0.3,
                spans 8-64), K=3 SAM drafts, T=1.0, bf16 logits N(0, sd 2) + 4
  draft_model   B=32, K=5, V=151936, fp32 target N(0, sd 2), draft logits =
                target + N(0,1), drafts sampled from softmax(draft/0.7), T=0.7
  long_rollout  B=256, Zipf(1.1) histories log-uniform in [16k, 32k] (copy prob
                0.5, spans 16-256), 512 steps extending by U{1..4} true tokens,
                K=3, greedy on bf16 logits
  sweep_b1024   B=1024, V=151936, K in {1,3,5,8}, fp32/bf16 N(0, sd 2), drafts
                uniform among each row's top-5, greedy and T=1.0
"""
from __future__ import annotations

import math

import numpy as np

V_LARGE = 151936


class ZipfTokens:
    """Zipf(a) over ranks 1..V truncated to V; token id = rank - 1."""

    def __init__(self, V: int, a: float = 1.1):
        w = 1.0 / np.arange(1, V + 1, dtype=np.float64) ** a
        self.cdf = np.cumsum(w)
        self.cdf /= self.cdf[-1]
        self.V = V

    def draw(self, rng: np.random.Generator, n: int) -> np.ndarray:
        u = rng.random(n)
        return np.minimum(np.searchsorted(self.cdf, u, side="right"), self.V - 1).astype(np.int32)


def make_stream(rng: np.random.Generator, n: int, V: int, p_copy: float, span_lo: int,
                span_hi: int, zipf: ZipfTokens | None = None) -> np.ndarray:
    """Token stream of length n built position by position: with probability
    p_copy (and when the stream is at least as long as the drawn span) copy a
    span of U[span_lo, span_hi] tokens from a uniformly chosen earlier start,
    otherwise draw one fresh token (uniform over V, or Zipf when given)."""
    out = np.empty(n, np.int32)
    pos = 0
    fresh_buf = np.empty(0, np.int32)
    fb = 0
    while pos < n:
        if rng.random() < p_copy:
            span = int(rng.integers(span_lo, span_hi + 1))
            if pos >= span:
                start = int(rng.integers(0, pos - span + 1))
                m = min(span, n - pos)
                out[pos:pos + m] = out[start:start + m]
                pos += m
                continue
        if fb >= fresh_buf.size:
            fresh_buf = (zipf.draw(rng, 4096) if zipf is not None
                         else rng.integers(0, V, size=4096, dtype=np.int32))
            fb = 0
        out[pos] = fresh_buf[fb]
        fb += 1
        pos += 1
    return out


def log_uniform_lengths(rng: np.random.Generator, B: int, lo: int, hi: int) -> np.ndarray:
    return np.exp(rng.uniform(math.log(lo), math.log(hi), size=B)).astype(np.int64).clip(lo, hi)


def gaussian_logits(rng: np.random.Generator, shape, sd: float) -> np.ndarray:
    return (rng.standard_normal(size=shape, dtype=np.float32) * np.float32(sd)).astype(np.float32)


def boost_truth(logits: np.ndarray, truth: np.ndarray, amount: float) -> None:
    """Add `amount` to logits[b, j, truth[b, j]] in place (truth < 0 skipped)."""
    B, R, _ = logits.shape
    for b in range(B):
        for j in range(R):
            t = int(truth[b, j])
            if t >= 0:
                logits[b, j, t] += np.float32(amount)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """fp32 values rounded to the nearest bf16 (ties to even), returned as
    fp32; NaN becomes the canonical quiet NaN.  The numpy twin of
    to_bf16(x).float()."""
    b = np.array(x, dtype=np.float32, copy=True).view(np.uint32)
    nan = (b & np.uint32(0x7FFFFFFF)) > np.uint32(0x7F800000)
    lsb = b >> np.uint32(16)
    lsb &= np.uint32(1)
    b += np.uint32(0x7FFF)
    b += lsb
    b &= np.uint32(0xFFFF0000)
    b[nan] = np.uint32(0x7FC00000)
    return b.view(np.float32)


def to_bf16(x: np.ndarray):
    """Round an fp32 array to a torch bfloat16 tensor (round-to-nearest-even)."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


# ------------------------------ workloads -----------------------------------

def tiny(seed: int = 1001, B: int = 4, V: int = 64, n: int = 256, K: int = 3):
    rng = np.random.default_rng(seed)
    streams = [make_stream(rng, n + K + 1, V, 0.3, 4, 16) for _ in range(B)]
    hist = np.stack([s[:n] for s in streams])
    truth = np.stack([s[n:n + K + 1] for s in streams])
    logits = gaussian_logits(rng, (B, K + 1, V), 1.0)
    boost_truth(logits, truth, 3.0)
    return dict(B=B, V=V, K=K, hist=hist, truth=truth, logits=logits, temperature=0.0)


def rs_bf16_b64(seed: int = 1002, B: int = 64, V: int = V_LARGE, n: int = 4096, K: int = 3,
                with_logits: bool = True):
    rng = np.random.default_rng(seed)
    z = ZipfTokens(V, 1.1)
    streams = [make_stream(rng, n + K + 1, V, 0.3, 8, 64, z) for _ in range(B)]
    hist = np.stack([s[:n] for s in streams])
    truth = np.stack([s[n:n + K + 1] for s in streams])
    out = dict(B=B, V=V, K=K, hist=hist, truth=truth, temperature=1.0)
    if with_logits:
        logits = gaussian_logits(rng, (B, K + 1, V), 2.0)
        boost_truth(logits, truth, 4.0)
        out["logits"] = logits  # fp32 values; the workload rounds them to bf16
    return out


def draft_model(seed: int = 1003, B: int = 32, V: int = V_LARGE, K: int = 5,
                T: float = 0.7, noise_sd: float = 1.0):
    """Target N(0, sd 2) [B, K+1, V]; draft = target[:, :K] + N(0, noise_sd);
    draft tokens sampled from softmax(draft / T) by the Gumbel-max trick."""
    rng = np.random.default_rng(seed)
    target = gaussian_logits(rng, (B, K + 1, V), 2.0)
    draftl = (target[:, :K] + gaussian_logits(rng, (B, K, V), noise_sd)).astype(np.float32)
    g = -np.log(-np.log(rng.random(size=(B, K, V))))
    drafts = np.argmax(draftl.astype(np.float64) / T + g, axis=-1).astype(np.int32)
    return dict(B=B, V=V, K=K, target=target, draft_logits=draftl, draft=drafts, temperature=T)


def long_rollout(seed: int = 1004, B: int = 256, V: int = V_LARGE, steps: int = 512, K: int = 3,
                 lo: int = 16384, hi: int = 32768):
    """Histories log-uniform in [lo, hi]; the stream continues for `steps`
    steps of U{1..4} tokens each (n_new[s, b])."""
    rng = np.random.default_rng(seed)
    z = ZipfTokens(V, 1.1)
    lens = log_uniform_lengths(rng, B, lo, hi)
    n_new = rng.integers(1, 5, size=(steps, B)).astype(np.int32)
    extra = n_new.sum(axis=0)
    streams = [make_stream(rng, int(lens[b] + extra[b]), V, 0.5, 16, 256, z) for b in range(B)]
    return dict(B=B, V=V, K=K, lens=lens.astype(np.int32), n_new=n_new, streams=streams,
                steps=steps, temperature=0.0)


def topk_drafts(logits_rows: np.ndarray, k: int, rng: np.random.Generator) -> np.ndarray:
    """For rows [..., V], a token drawn uniformly among each row's top-k."""
    top = np.argpartition(-logits_rows, k - 1, axis=-1)[..., :k]
    pick = rng.integers(0, k, size=top.shape[:-1])
    return np.take_along_axis(top, pick[..., None], axis=-1)[..., 0].astype(np.int32)


def sweep_host(seed: int, B: int, K: int, V: int = V_LARGE):
    """Host-side sweep inputs (for sizes the host can hold comfortably)."""
    rng = np.random.default_rng(seed)
    logits = gaussian_logits(rng, (B, K + 1, V), 2.0)
    drafts = topk_drafts(logits[:, :K], 5, rng)
    return logits, drafts


def sweep_device(seed: int, B: int, K: int, V: int, dtype, device):
    """Device-side sweep inputs for the full B=1024 sizes: N(0, sd 2) logits
    from a seeded torch generator on `device`, drafts uniform among each row's
    top-5.  Returns (logits [B, K+1, V] of `dtype`, drafts [B, K] int32)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    logits = torch.empty((B, K + 1, V), dtype=torch.float32, device=device)
    for b0 in range(0, B, 64):  # bounded temporaries
        logits[b0:b0 + 64].normal_(0.0, 2.0, generator=g)
    logits = logits.to(dtype)
    top = torch.topk(logits[:, :K].float(), 5, dim=-1).indices
    pick = torch.randint(0, 5, (B, K, 1), device=device, generator=g)
    drafts = torch.gather(top, -1, pick)[..., 0].to(torch.int32).contiguous()
    return logits.contiguous(), drafts


def draft_model_device(seed: int, B: int, K: int, V: int, T: float, device, noise_sd: float = 1.0):
    """The draft-model workload drawn on `device` from a seeded torch
    generator (the same distributions as draft_model): target N(0, sd 2)
    [B, K+1, V] fp32, draft logits = target[:, :K] + N(0, noise_sd), draft
    tokens sampled from softmax(draft / T) by the Gumbel-max trick."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    target = torch.empty((B, K + 1, V), dtype=torch.float32, device=device).normal_(0.0, 2.0, generator=g)
    noise = torch.empty((B, K, V), dtype=torch.float32, device=device).normal_(0.0, noise_sd, generator=g)
    draftl = (target[:, :K] + noise).contiguous()
    u = torch.rand((B, K, V), dtype=torch.float64, device=device, generator=g).clamp_min(1e-300)
    drafts = torch.argmax(draftl.double() / T - torch.log(-torch.log(u)), dim=-1).to(torch.int32)
    return target.contiguous(), draftl, drafts.contiguous()


def sweep_host_bf16(seed: int, B: int, K: int, V: int = V_LARGE):
    """Host sweep inputs rounded to bf16 (returned as the exact fp32 values),
    drafts uniform among each rounded row's top-5."""
    rng = np.random.default_rng(seed)
    logits = to_bf16(gaussian_logits(rng, (B, K + 1, V), 2.0)).float().numpy()
    drafts = topk_drafts(logits[:, :K], 5, rng)
    return logits, drafts
