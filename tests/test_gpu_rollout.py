"""The decode step (verify, extend, draft in one call) and the rollout loop
with the adaptive switch, on a toy target model whose logits depend on the
position only: losslessness against plain decoding (greedy) and against an
oracle-driven rollout (sampling)."""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ss(cuda_device):
    import sam_drafting_verification_gb300 as ss
    return ss


class ToyModel:
    """logits(row b, position p) = noise[(b * 7919 + p) % P] + boost at truth[b, p]."""

    def __init__(self, truth, V, boost, sd, seed, dev, P=257):
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        self.noise = torch.empty((P, V), device=dev).normal_(0.0, sd, generator=g)
        self.truth = torch.as_tensor(np.asarray(truth, np.int64), device=dev)
        self.boost, self.P, self.V = boost, P, V

    def logits_at(self, rows, pos):  # rows, pos: int64 [m]
        x = self.noise[(rows * 7919 + pos) % self.P].clone()
        if self.boost:
            t = self.truth[rows, pos.clamp(max=self.truth.shape[1] - 1)]
            x[torch.arange(x.shape[0], device=x.device), t] += self.boost
        return x

    def __call__(self, rows, n_done, draft, draft_len):
        n, K = draft.shape
        r = rows.long().repeat_interleave(K + 1)
        p = (n_done.view(-1, 1) + torch.arange(K + 1, device=rows.device).view(1, -1)).reshape(-1)
        return self.logits_at(r, p).view(n, K + 1, self.V).contiguous()


def _i32(a, dev):
    return torch.as_tensor(np.ascontiguousarray(a, dtype=np.int32), device=dev)


def test_spec_step_matches_separate_calls(ss, cuda_device):
    rng = np.random.default_rng(3)
    B, V, K, n0 = 24, 3000, 3, 400
    hist = np.stack([workloads.make_stream(rng, n0, V, 0.5, 4, 32) for _ in range(B)]).astype(np.int32)
    a = ss.SamBatch(B, 1000, V, device=cuda_device)
    b = ss.SamBatch(B, 1000, V, device=cuda_device)
    for x in (a, b):
        x.extend(_i32(hist, cuda_device), _i32(np.full(B, n0), cuda_device))
    draft, dlen, _, _ = a.draft(K)
    rows = torch.as_tensor(rng.permutation(B)[:17].astype(np.int32), device=cuda_device)
    d_sub, dl_sub = draft[rows.long()].contiguous(), dlen[rows.long()].contiguous()
    logits = torch.from_numpy(workloads.gaussian_logits(rng, (17, K + 1, V), 2.0)).to(cuda_device)
    for T in (0.0, 1.0):
        r = a.spec_step(logits, d_sub, dl_sub, K_next=4, rows=rows, temperature=T, seed=7, step=2)
        v = ss.spec_verify(logits, d_sub, dl_sub, temperature=T, seed=7, step=2, emit=True)
        d2, dl2, ml2, me2 = b.step_rows(rows, v["emit"], v["emit_len"], 4)
        for k in ("accept_len", "out_token", "emit", "emit_len", "status"):
            assert torch.equal(r[k], v[k]), k
        assert torch.equal(r["next_draft"], d2) and torch.equal(r["next_draft_len"], dl2)
        assert torch.equal(r["match_len"], ml2) and torch.equal(r["min_endpos"], me2)
        d_sub, dl_sub = r["next_draft"][:, :K].contiguous(), r["next_draft_len"].clamp(max=K).contiguous()
    for i in range(B):
        x, y = a.dump(i), b.dump(i)
        for k in ("len", "link", "min_endpos", "edges"):
            np.testing.assert_array_equal(x[k], y[k])
    # K = 0: plain decoding of the bonus row, automata extended by one token
    lg0 = logits[:, :1].contiguous()
    r0 = a.spec_step(lg0, torch.zeros((17, 0), dtype=torch.int32, device=cuda_device), None,
                     K_next=0, rows=rows, temperature=1.0, seed=7, step=3)
    assert (r0["accept_len"] == 0).all() and (r0["emit_len"] == 1).all()
    assert (r0["next_draft_len"] == 0).all()


def _truth_streams(B, V, n, seed):
    rng = np.random.default_rng(seed)
    return np.stack([workloads.make_stream(rng, n, V, 0.5, 8, 32) for _ in range(B)]).astype(np.int64)


def test_greedy_rollout_is_lossless_and_switches(ss, cuda_device):
    from sam_drafting_verification_gb300.rollout import Rollout, speculation_k
    B, V, P0 = 12, 2000, 64
    truth = _truth_streams(B, V, 600, 11)
    limits = [40 + 37 * b for b in range(B)]  # uneven lengths: a long tail
    model = ToyModel(truth[:, P0:], V, boost=60.0, sd=2.0, seed=5, dev=cuda_device)
    runs = {}
    for name, K, thr in (("plain", 0, None), ("spec", 3, None), ("switch", 3, 4)):
        batch = ss.SamBatch(B, 1200, V, device=cuda_device)
        batch.extend(_i32(truth[:, :P0], cuda_device), _i32(np.full(B, P0), cuda_device))
        res = Rollout(batch, model, K=K, threshold=thr, temperature=0.0).run(limits)
        for b in range(B):
            assert res.tokens[b] == truth[b, P0:P0 + limits[b]].tolist(), (name, b)
        runs[name] = res
    assert runs["spec"].steps < runs["plain"].steps and runs["spec"].accepted > 0
    sw = runs["switch"]
    # each step drafted with the policy of the step before it
    for i in range(1, sw.steps):
        assert sw.k_per_step[i] == speculation_k(sw.active_per_step[i - 1], 4, 3)
    assert 0 in sw.k_per_step and 3 in sw.k_per_step
    assert runs["plain"].steps <= max(limits) and all(k == 0 for k in runs["plain"].k_per_step)


def test_sampling_rollout_matches_oracle_rollout(ss, cuda_device):
    """T = 1 on a small vocabulary: the rollout through the library and the
    same loop through the oracle's automata and verification emit the same
    tokens (coins keyed by the sequence's index in each step's call)."""
    from sam_drafting_verification_gb300.rollout import Rollout, speculation_k
    B, V, P0, K, thr, T, seed = 6, 64, 48, 3, 3, 1.0, 99
    truth = _truth_streams(B, V, 400, 21)
    limits = [30 + 20 * b for b in range(B)]
    model = ToyModel(truth[:, P0:], V, boost=3.0, sd=1.0, seed=8, dev=cuda_device)
    batch = ss.SamBatch(B, 800, V, device=cuda_device)
    batch.extend(_i32(truth[:, :P0], cuda_device), _i32(np.full(B, P0), cuda_device))
    res = Rollout(batch, model, K=K, threshold=thr, temperature=T, seed=seed).run(limits)

    # the same loop with the oracle
    sams = [oracle.Sam(V) for _ in range(B)]
    for b in range(B):
        sams[b].extend(truth[b, :P0])
    out = [[] for _ in range(B)]
    active = list(range(B))
    k = speculation_k(len(active), thr, K)
    drafts = {b: sams[b].draft(k)[:2] if k else (np.zeros(0, np.int32), 0) for b in active}
    step = 0
    while active:
        n = len(active)
        kk = len(drafts[active[0]][0])
        d = np.stack([np.maximum(drafts[b][0], 0) for b in active]).reshape(n, kk).astype(np.int32)
        dl = np.array([drafts[b][1] for b in active], np.int32)
        rows = torch.tensor(active, dtype=torch.int32, device=cuda_device)
        n_done = torch.tensor([len(out[b]) for b in active], dtype=torch.int64, device=cuda_device)
        lg = model(rows, n_done, torch.as_tensor(d, device=cuda_device), torch.as_tensor(dl, device=cuda_device))
        o = oracle.verify(lg.cpu().numpy(), d, dl, temperature=T, seed=seed, step=step)
        k_next = speculation_k(n, thr, K)
        keep = []
        for i, b in enumerate(active):
            L = int(o["accept_len"][i])
            toks = list(d[i, :L]) + [int(o["out_token"][i])]
            sams[b].extend(np.asarray(toks, np.int32))
            room = limits[b] - len(out[b])
            out[b].extend(int(t) for t in toks[:room])
            if len(out[b]) < limits[b]:
                keep.append(b)
            drafts[b] = sams[b].draft(k_next)[:2] if k_next else (np.zeros(0, np.int32), 0)
        active = keep
        step += 1
    assert res.steps == step
    for b in range(B):
        assert res.tokens[b] == out[b], b
