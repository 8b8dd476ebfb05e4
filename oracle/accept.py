"""Oracle of tree acceptance and KV compaction.

The pages fix the contract: keep drafted tokens from the root while they pass
the acceptance test, which is equality with the target's choice under greedy
decoding, or the rejection-sampling rule under sampling; at the first rejection
use the target's own token, so every cycle gains at least one token and the
output distribution is exactly the target's ("EAGLE: Feature-Level Drafting",
"Speculative decoding in four moves", items 3-4; "EAGLE-2: Context-Aware
Dynamic Draft Trees", section "The Mask Preserves Tree Semantics in One Target
Pass": strict speculative sampling selects and corrects a branch; table
"Putting It Together", step 5). The multi-candidate sampling rule is not
spelled out on the pages. The reading used here is recursive point-mass
rejection: at node u with target distribution p, try the kept children in
their draft-rank order and accept child t with probability
p(t) / (1 - sum of p over the children already tried); if every child is
rejected (or u is a leaf) the bonus token is drawn from p restricted to the
vocabulary minus those children, renormalised. Each token then has marginal
probability p(t), so the rule is lossless for deterministically chosen
children. The bonus draw is a Gumbel-argmax of log p over the allowed set.

KV compaction is implied by "lossless committed tokens and the next verified
state" (EAGLE-2 page, "Putting It Together", step 5): the accepted rows' K/V,
written at scratch slots n + row during the verify pass, move to slots
n + 1 .. n + L. K is stored after RoPE at position n + depth = n + j, its final
position, so the move is a pure copy.

Test infrastructure: only tests, the smoke check and the bench's CPU baseline
use this package.
"""
from __future__ import annotations

from typing import Callable, List, Sequence, Tuple

import numpy as np

from .tree import FlatTree


def argmax_lowest(v: np.ndarray) -> int:
    """argmax with ties to the lowest index."""
    v = np.asarray(v)
    return int(np.flatnonzero(v == v.max())[0])


def greedy_walk(tree: FlatTree, target_argmax: Sequence[int]) -> Tuple[List[int], int]:
    """Greedy acceptance. Returns (accepted rows in path order, bonus token)."""
    u = 0
    path: List[int] = []
    while True:
        a = int(target_argmax[u])
        nxt = [v for v in tree.children(u) if int(tree.token[v]) == a]
        if not nxt:
            return path, a
        u = nxt[0]
        path.append(u)


def accept_threshold_test(u: float, tried: float, pt: float, dtype=np.float32) -> bool:
    """Accept iff u * (1 - tried) < p(t) (equivalently u < p(t) / (1 - tried) when the
    residual mass is positive; with no residual mass left any child with p(t) > 0 is taken)."""
    d = dtype
    return bool(d(u) * (d(1.0) - d(tried)) < d(pt))


def sample_walk(tree: FlatTree, p_child: Callable[[int, int], float],
                uniform: Callable[[int, int], float],
                bonus: Callable[[int, List[int]], int], dtype=np.float32) -> Tuple[List[int], int]:
    """Point-mass rejection walk. p_child(row, token) = target probability of `token` at
    `row`; uniform(row, i) = the draw for the i-th tried child of `row`; bonus(row, excluded
    tokens) = the token drawn from p restricted to the rest. The running sum of tried mass
    and the threshold test use `dtype` arithmetic."""
    u = 0
    path: List[int] = []
    while True:
        tried = dtype(0.0)
        taken = None
        kids = tree.children(u)
        for i, v in enumerate(kids):
            pt = dtype(p_child(u, int(tree.token[v])))
            if accept_threshold_test(uniform(u, i), tried, pt, dtype):
                taken = v
                break
            tried = dtype(tried + pt)
        if taken is None:
            return path, bonus(u, [int(tree.token[v]) for v in kids])
        path.append(taken)
        u = taken


def enumerate_walk(tree: FlatTree, probs: np.ndarray) -> List[Tuple[List[int], int, float]]:
    """Every outcome of the point-mass rejection walk with its exact probability.
    probs [m+1, V]: the target distribution at each flattened row. Returns
    [(accepted rows, bonus token, probability)]."""
    out: List[Tuple[List[int], int, float]] = []

    def rec(u: int, path: List[int], w: float):
        p = probs[u]
        kids = tree.children(u)
        tried = 0.0
        reach = w
        for v in kids:
            pt = float(p[int(tree.token[v])])
            resid = 1.0 - tried
            a = 1.0 if resid <= 0.0 else min(1.0, pt / resid)
            if reach * a > 0.0:
                rec(v, path + [v], reach * a)
            reach *= (1.0 - a)
            tried += pt
        if reach > 0.0:
            excluded = {int(tree.token[v]) for v in kids}
            rest = 1.0 - sum(float(p[t]) for t in excluded)
            if rest > 0.0:
                for t in range(p.shape[0]):
                    if t not in excluded and p[t] > 0.0:
                        out.append((path, t, reach * float(p[t]) / rest))

    rec(0, [], 1.0)
    return out


def compact(k: np.ndarray, v: np.ndarray, n: int, path_rows: Sequence[int]) -> None:
    """In-place KV compaction over all layers: slot n + j <- slot n + path_rows[j-1],
    j = 1..L. k, v: [layers, n_kv, capacity, d]. All sources are read before any write."""
    if not len(path_rows):
        return
    src = [n + int(r) for r in path_rows]
    ks = k[:, :, src, :].copy()
    vs = v[:, :, src, :].copy()
    dst = list(range(n + 1, n + 1 + len(src)))
    k[:, :, dst, :] = ks
    v[:, :, dst, :] = vs
