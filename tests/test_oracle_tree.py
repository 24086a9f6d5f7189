"""Pins of the oracle's tree verification (gogongxt.com notes "投机采样",
SGLang 的实现: candidates tried sibling by sibling against one coin per
depth; rejected candidates removed before the final sample):
  * a tree whose nodes have one child each is the linear chain of drafts:
    identical to the (separately pinned) linear verification;
  * greedy trees follow numpy's argmax down the tree;
  * losslessness: the first emitted token follows the root row's softmax and,
    after an accepted child, the second follows that child's row (chi-square);
  * malformed trees are refused."""
import numpy as np
import pytest
from scipy import special, stats

import oracle
import workloads


def _chain(draft):
    """Tree arrays of a linear draft d_0 .. d_{K-1}: node n + 1 holds d_n."""
    K = len(draft)
    tok = np.concatenate([[-1], draft]).astype(np.int32)
    fc = np.array([n + 1 if n < K else -1 for n in range(K + 1)], np.int32)
    ns = np.full(K + 1, -1, np.int32)
    return tok, fc, ns


@pytest.mark.parametrize("T", [0.0, 0.7, 1.0])
def test_chain_trees_equal_linear_verification(T):
    rng = np.random.default_rng(int(T * 10) + 3)
    B, K, V = 40, 4, 50
    logits = workloads.gaussian_logits(rng, (B, K + 1, V), 1.5)
    draft = np.argsort(-logits[:, :K], axis=-1)[..., :3][np.arange(B)[:, None], np.arange(K)[None, :],
                                                         rng.integers(0, 3, (B, K))].astype(np.int32)
    lin = oracle.verify(logits, draft, None, temperature=T, seed=5, step=2)
    trees = [_chain(draft[b]) for b in range(B)]
    tok, fc, ns = (np.stack([t[i] for t in trees]) for i in range(3))
    tr = oracle.tree_verify(logits, tok, fc, ns, temperature=T, seed=5, step=2)
    assert (tr["status"] == 0).all()
    np.testing.assert_array_equal(tr["accept_len"], lin["accept_len"])
    np.testing.assert_array_equal(tr["out_token"], lin["out_token"])
    for b in range(B):
        L = tr["accept_len"][b]
        assert list(tr["path"][b, :L]) == list(range(1, L + 1)) and (tr["path"][b, L:] == -1).all()


def _sample_tree():
    # node: 0 root; 1,2,3 children of 0 (tokens 2, 4, 1); 4,5 children of 1
    # (tokens 0, 3); 6 child of 2 (token 5)
    tok = np.array([-1, 2, 4, 1, 0, 3, 5], np.int32)
    fc = np.array([1, 4, 6, -1, -1, -1, -1], np.int32)
    ns = np.array([-1, 2, 3, -1, 5, -1, -1], np.int32)
    return tok, fc, ns


def test_greedy_follows_argmax():
    rng = np.random.default_rng(8)
    tok, fc, ns = _sample_tree()
    N, V, B = len(tok), 6, 300
    logits = workloads.gaussian_logits(rng, (B, N, V), 2.0)
    # make some argmaxes hit the tree
    logits[::2, 0, 2] += 6.0
    logits[::4, 1, 3] += 6.0
    tr = oracle.tree_verify(logits, np.tile(tok, (B, 1)), np.tile(fc, (B, 1)), np.tile(ns, (B, 1)), 0.0)
    for b in range(B):
        cur, depth = 0, 0
        while True:
            a = int(np.argmax(logits[b, cur]))
            nxt = [c for c in _children(fc, ns, cur) if tok[c] == a]
            if not nxt:
                break
            cur = nxt[0]
            assert tr["path"][b, depth] == cur
            depth += 1
        assert tr["accept_len"][b] == depth and tr["out_token"][b] == a


def _children(fc, ns, n):
    out, c = [], fc[n]
    while c != -1:
        out.append(c)
        c = ns[c]
    return out


def test_sampled_tokens_follow_the_target():
    rng = np.random.default_rng(12)
    tok, fc, ns = _sample_tree()
    N, V, B, T = len(tok), 6, 200000, 1.0
    rows = workloads.gaussian_logits(rng, (N, V), 1.0)
    logits = np.broadcast_to(rows, (B, N, V)).copy()
    tr = oracle.tree_verify(logits, np.tile(tok, (B, 1)), np.tile(fc, (B, 1)), np.tile(ns, (B, 1)), T,
                            seed=31, step=4)
    assert (tr["status"] == 0).all()
    L, out, path = tr["accept_len"], tr["out_token"], tr["path"]
    first = np.where(L >= 1, tok[np.maximum(path[:, 0], 0)], out)
    p0 = special.softmax(rows[0].astype(np.float64) / T)
    pvals = [stats.chisquare(np.bincount(first, minlength=V), p0 * B).pvalue]
    # after accepting child 1 (token 2) at depth 0, the second token follows row 1
    sel = (L >= 1) & (path[:, 0] == 1)
    second = np.where(L[sel] >= 2, tok[np.maximum(path[sel, 1], 0)], out[sel])
    p1 = special.softmax(rows[1].astype(np.float64) / T)
    pvals.append(stats.chisquare(np.bincount(second, minlength=V), p1 * sel.sum()).pvalue)
    assert min(pvals) > 1e-3 / len(pvals), pvals


def test_malformed_trees_are_refused():
    tok, fc, ns = _sample_tree()
    V, N = 6, len(tok)
    logits = np.zeros((1, N, V), np.float32)
    cases = []
    t2 = tok.copy(); t2[2] = 2; cases.append((t2, fc, ns))            # equal sibling tokens
    f2 = fc.copy(); f2[4] = 1; cases.append((tok, f2, ns))             # link to a smaller index
    n2 = ns.copy(); n2[5] = 6; cases.append((tok, fc, n2))             # node 6 linked twice
    t3 = tok.copy(); t3[3] = V; cases.append((t3, fc, ns))             # token out of range
    n3 = ns.copy(); n3[0] = 2; cases.append((tok, fc, n3))             # the root has a sibling
    for t, f, n in cases:
        tr = oracle.tree_verify(logits, t[None], f[None], n[None], 1.0)
        assert tr["status"][0] == 6 and tr["accept_len"][0] == -1


def test_node_info_closed_form():
    # uniform row over 4 tokens, children {1, 2}: running sums 1/4, 1/2; the
    # final distribution keeps tokens 0 and 3 with mass 1/2 each
    acc, lo, hi, mass = oracle.tree_node_info(np.zeros(4, np.float32), 1.0, [1, 2], 3)
    np.testing.assert_allclose(acc, [0.25, 0.5])
    assert (lo, hi, mass) == (0.5, 1.0, 0.5)
