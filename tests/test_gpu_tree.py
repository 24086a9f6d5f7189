"""Tree verification on the GPU against the oracle: accepted paths, emitted
tokens and statuses; sampling decisions identical up to the excused band
(a coin within 1e-6 of a child's running-sum threshold, or of a boundary of
the oracle's interval of the GPU's token)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import compare_trees

pytestmark = pytest.mark.gpu

BAND = 1e-6


@pytest.fixture(scope="module")
def ss(cuda_device):
    import sam_drafting_verification_gb300 as ss
    return ss


def random_trees(rng, logits, N, width):
    """Per sequence a tree of N nodes: node n >= 1 hangs under a random earlier
    node (at most `width` children each); its token is one of its parent
    row's 8 most likely tokens, distinct among siblings."""
    B = logits.shape[0]
    tok = np.full((B, N), -1, np.int32)
    fc = np.full((B, N), -1, np.int32)
    ns = np.full((B, N), -1, np.int32)
    for b in range(B):
        kids = {0: []}
        for n in range(1, N):
            cands = [p for p in kids if len(kids[p]) < width]
            par = int(rng.choice(cands))
            top = list(np.argsort(-logits[b, par])[:8])
            used = {int(tok[b, c]) for c in kids[par]}
            choice = [t for t in top if int(t) not in used]
            tok[b, n] = int(choice[int(rng.integers(0, len(choice)))])
            if kids[par]:
                ns[b, kids[par][-1]] = n
            else:
                fc[b, par] = n
            kids[par].append(n)
            kids[n] = []
    return tok, fc, ns


@pytest.mark.parametrize("T", [0.0, 0.7, 1.0])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_random_trees(ss, cuda_device, T, dtype):
    rng = np.random.default_rng(int(T * 10) + (7 if dtype == torch.bfloat16 else 0))
    B, N, V = 48, 12, 40000
    logits = workloads.gaussian_logits(rng, (B, N, V), 2.0)
    tok, fc, ns = random_trees(rng, logits, N, 3)
    tt = torch.from_numpy(logits).to(dtype)
    rows = tt.float().numpy()
    i32 = lambda a: torch.as_tensor(a, device=cuda_device)  # noqa: E731
    g = ss.spec_verify_tree(tt.to(cuda_device), i32(tok), i32(fc), i32(ns), temperature=T, seed=21,
                            step=3, debug=True)
    g = {k: v.cpu().numpy() for k, v in g.items()}
    o = oracle.tree_verify(rows, tok, fc, ns, temperature=T, seed=21, step=3)
    compare_trees(g, o, rows, tok, fc, ns, T, seed=21, step=3)
    if T == 0.0:
        assert (g["accept_len"] > 0).any()


def test_chain_trees_equal_linear_kernel(ss, cuda_device):
    rng = np.random.default_rng(5)
    B, K, V = 64, 4, 30000
    logits, draft = workloads.sweep_host(77, B, K, V)
    am = np.argmax(logits[:, :K], axis=-1).astype(np.int32)
    draft[::2] = am[::2]
    tok = np.concatenate([np.full((B, 1), -1), draft], 1).astype(np.int32)
    fc = np.tile(np.array([n + 1 if n < K else -1 for n in range(K + 1)], np.int32), (B, 1))
    ns = np.full((B, K + 1), -1, np.int32)
    lg = torch.from_numpy(logits).to(cuda_device)
    i32 = lambda a: torch.as_tensor(a, device=cuda_device)  # noqa: E731
    for T in (0.0, 1.0):
        t = ss.spec_verify_tree(lg, i32(tok), i32(fc), i32(ns), temperature=T, seed=9, step=1)
        lin = ss.spec_verify(lg, i32(draft), None, temperature=T, seed=9, step=1, emit=True)
        assert torch.equal(t["accept_len"], lin["accept_len"])
        assert torch.equal(t["out_token"], lin["out_token"])
        assert torch.equal(t["emit"], lin["emit"])


def test_malformed_trees(ss, cuda_device):
    V, N = 100, 5
    tok = np.array([[-1, 3, 4, 5, 6]] * 4, np.int32)
    fc = np.array([[1, 3, -1, -1, -1]] * 4, np.int32)
    ns = np.array([[-1, 2, -1, 4, -1]] * 4, np.int32)
    tok[1, 2] = 3          # equal sibling tokens
    fc[2, 1] = 1           # a node linked to itself
    tok[3, 4] = V          # token out of range
    lg = torch.zeros((4, N, V), device=cuda_device)
    i32 = lambda a: torch.as_tensor(a, device=cuda_device)  # noqa: E731
    r = ss.spec_verify_tree(lg, i32(tok), i32(fc), i32(ns), temperature=1.0)
    st = r["status"].cpu().numpy()
    assert st[0] == 0 and list(st[1:]) == [6, 6, 6]
    o = oracle.tree_verify(lg.cpu().numpy(), tok, fc, ns, temperature=1.0)
    assert list(o["status"]) == list(st)
