"""Host loop of a speculative rollout over the library's decode step.

Each step drafts with the sequences' suffix automata and verifies the drafts
against the target model's logits in one `sam_spec_step` call ("SAM投机推理：
长序列强化学习训练加速利器" §1.1).  Whether a step speculates follows the
adaptive switch of the same article, §3.1.1: drafting is on only while the
number of active requests is at most a threshold (late in a rollout, when a
few long requests are left).

The loop keeps the active set on the host (it reads each step's emitted
tokens back to detect finished sequences); everything per token runs in the
library's kernels.  The target model is a callable:

    model(rows, n_done, draft, draft_len) -> logits [n, K+1, V]

with rows (int32 [n], the automata / sequences of this step), n_done (int64
[n], tokens each has generated so far), draft (int32 [n, K]) and draft_len
(int32 [n]); row j of a sequence's logits scores the token after its first j
drafts.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

from . import SamBatch, verify_workspace


def speculation_k(n_active: int, threshold: int | None, K: int) -> int:
    """Draft length for a step with n_active requests: K while n_active is at
    most the threshold (no threshold: always), else 0 (plain decoding)."""
    if threshold is None or n_active <= threshold:
        return int(K)
    return 0


@dataclass
class RolloutResult:
    tokens: list                      # generated tokens per sequence (python ints)
    steps: int = 0                    # decode steps run
    k_per_step: list = field(default_factory=list)       # draft length used by each step
    active_per_step: list = field(default_factory=list)  # active sequences at each step
    accepted: int = 0                 # drafts accepted over the rollout


class Rollout:
    def __init__(self, batch: SamBatch, model, K: int = 3, threshold: int | None = None,
                 temperature: float = 0.0, seed: int = 0, eos: int | None = None):
        self.batch, self.model, self.K = batch, model, int(K)
        self.threshold, self.temperature, self.seed, self.eos = threshold, float(temperature), int(seed), eos

    def run(self, max_new_tokens) -> RolloutResult:
        """Generates up to max_new_tokens[b] tokens per sequence (or until eos)
        from the automata's current texts (prompts already extended).

        The step that finishes a sequence extends its automaton by every token
        that step emitted, so the automaton may hold up to K tokens beyond the
        ones returned for it (those after its eos or past its limit).  A
        finished sequence's automaton is not used again by this rollout; a
        caller that goes on with it should reset and rebuild it from the
        returned text."""
        dev = self.batch.device
        B = self.batch.B
        limit = [int(x) for x in max_new_tokens]
        out = [[] for _ in range(B)]
        active = [b for b in range(B) if limit[b] > 0]
        res = RolloutResult(tokens=out)
        if not active:
            return res
        rows = torch.tensor(active, dtype=torch.int32, device=dev)
        k = speculation_k(len(active), self.threshold, self.K)
        empty = torch.zeros((len(active), 0), dtype=torch.int32, device=dev)
        zero = torch.zeros(len(active), dtype=torch.int32, device=dev)
        # the first drafts: an empty extension that drafts k tokens
        draft, dlen, _, _ = self.batch.step_rows(rows, empty, zero, k)
        # one workspace for the whole rollout, and one buffer for the per-step
        # outputs the host reads (emit, emit_len, status, accept_len), so that
        # a step costs one device-to-host copy
        ws = verify_workspace(len(active), self.K, 1, dev)
        hostbuf = torch.empty(len(active) * (self.K + 4), dtype=torch.int32, device=dev)
        step = 0
        while active:
            n = len(active)
            n_done = torch.tensor([len(out[b]) for b in active], dtype=torch.int64, device=dev)
            logits = self.model(rows, n_done, draft, dlen)
            k_next = speculation_k(n, self.threshold, self.K)
            K1 = int(draft.shape[1]) + 1
            o = {"emit": hostbuf[:n * K1].view(n, K1), "emit_len": hostbuf[n * K1:n * K1 + n],
                 "status": hostbuf[n * K1 + n:n * K1 + 2 * n],
                 "accept_len": hostbuf[n * K1 + 2 * n:n * K1 + 3 * n]}
            r = self.batch.spec_step(logits, draft, dlen, K_next=k_next, rows=rows,
                                     temperature=self.temperature, seed=self.seed, step=step,
                                     workspace=ws, out=o)
            res.k_per_step.append(int(draft.shape[1]))
            res.active_per_step.append(n)
            h = hostbuf[:n * K1 + 3 * n].cpu()
            emit = h[:n * K1].view(n, K1).tolist()
            elen = h[n * K1:n * K1 + n].tolist()
            st = h[n * K1 + n:n * K1 + 2 * n].tolist()
            acc = h[n * K1 + 2 * n:n * K1 + 3 * n].tolist()
            keep = []
            for i, b in enumerate(active):
                if st[i] != 0:
                    raise RuntimeError(f"sequence {b}: verification status {st[i]}")
                res.accepted += acc[i]
                toks = emit[i][:elen[i]]
                room = limit[b] - len(out[b])
                stop = False
                for t in toks[:room]:
                    out[b].append(t)
                    if self.eos is not None and t == self.eos:
                        stop = True
                        break
                if not stop and len(out[b]) < limit[b]:
                    keep.append(i)
            step += 1
            res.steps = step
            if len(keep) != n:
                idx = torch.tensor(keep, dtype=torch.int64, device=dev)
                active = [active[i] for i in keep]
                rows = rows[idx].contiguous()
                draft = r["next_draft"][idx].contiguous()
                dlen = r["next_draft_len"][idx].contiguous()
            else:
                draft, dlen = r["next_draft"], r["next_draft_len"]
        return res
