"""Oracle of the EAGLE-2 dynamic draft tree.

Steps, in the order the pages give them:
- path value V_i = product of the draft confidences c_j on the root-to-node path
  ("EAGLE-2: Context-Aware Dynamic Draft Trees", section "Path Value Ranks
  Prefixes, Not Isolated Tokens", the V_i equation; "EAGLE 三代", §3, s(v));
  ranked in log space to avoid underflow (same EAGLE-2 page, table "Where It
  Breaks", row "Prefix-product underflow");
- expansion: at each depth the top-k current leaves by V are expanded in one
  drafter call (EAGLE-2 page, same section; "EAGLE: Feature-Level Drafting",
  list "How EAGLE-2 builds its tree", items 1-2);
- rerank: keep the m best of all generated nodes, preferring shallower nodes on
  ties, which gives a connected tree (EAGLE-2 page, section "Global Reranking
  Separates Exploration from Verification"; "EAGLE: Feature-Level Drafting",
  "Worked example, step by step");
- flatten + ancestry mask: each flattened row sees the root, itself and its
  ancestors, never a sibling branch (EAGLE-2 page, section "The Mask Preserves
  Tree Semantics in One Target Pass", Figure 7).

Readings where the pages are silent: log V is an fp32 running sum
log V_child = fp32(log V_parent + log c_child); a node's k children are its
drafter's top-k tokens by (logit desc, token id asc); expansion picks nodes by
(log V desc, generation index asc); the rerank key is (log V desc, depth asc,
generation index asc); generation indices run depth-major, children of the
r-th expanded node (in selection order) in their top-k rank order.

Static tree (EAGLE-1): the tree has the same shape every cycle, decided in
advance ("EAGLE: Feature-Level Drafting", section "EAGLE-2 and dynamic draft
trees"; "EAGLE-2" page, section "Why This Exists"). Reading, as the pages give no
shape: a topology of nodes (parent, rank), rank r naming the drafter's r-th best
child of the parent (depth-1 nodes: the root's r-th candidate). The same machinery
draws it: at each depth the k expansion rows are the topology's nodes that have
children, in topology order, then (to keep k rows per depth) the lowest-index
other nodes of that depth; the kept set is the topology's nodes, with no rerank.
A chain is the topology with one rank-0 child per depth.

Test infrastructure: only tests, the smoke check and the bench's CPU baseline
use this package.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Sequence, Tuple

import numpy as np

F32 = np.float32


def topk_ids(values: np.ndarray, k: int, exclude: Sequence[int] = ()) -> np.ndarray:
    """Indices of the k largest values, ties to the lower index; `exclude` ids skipped."""
    v = np.asarray(values, dtype=np.float64).copy()
    if len(exclude):
        v[np.asarray(list(exclude), dtype=np.int64)] = -np.inf
    order = np.lexsort((np.arange(v.shape[0]), -v))
    return order[:k]


@dataclass
class NodeTable:
    token: List[int] = field(default_factory=list)
    parent: List[int] = field(default_factory=list)   # node index, -1 = the root
    depth: List[int] = field(default_factory=list)
    logv: List[np.float32] = field(default_factory=list)

    def __len__(self):
        return len(self.token)

    def add(self, token: int, parent: int, logc: float) -> int:
        base = F32(0.0) if parent < 0 else self.logv[parent]
        self.token.append(int(token))
        self.parent.append(int(parent))
        self.depth.append(1 if parent < 0 else self.depth[parent] + 1)
        self.logv.append(F32(base + F32(logc)))
        return len(self.token) - 1

    def path(self, i: int) -> List[int]:
        """Node indices from depth 1 down to node i."""
        out = []
        while i >= 0:
            out.append(i)
            i = self.parent[i]
        return out[::-1]


def select_expand(t: NodeTable, depth: int, k: int) -> List[int]:
    """The k nodes of `depth` with the largest (log V, -generation index)."""
    cand = [i for i in range(len(t)) if t.depth[i] == depth]
    cand.sort(key=lambda i: (-float(t.logv[i]), i))
    return cand[:k]


def rerank(t: NodeTable, m: int) -> List[int]:
    """Global top-m of all generated nodes by (log V desc, depth asc, generation asc)."""
    idx = list(range(len(t)))
    idx.sort(key=lambda i: (-float(t.logv[i]), t.depth[i], i))
    return idx[:m]


@dataclass
class FlatTree:
    """Flattened tree: row 0 = root, rows 1.. = kept nodes in generation order."""
    token: np.ndarray     # int [m+1]
    parent: np.ndarray    # int [m+1], flattened index of the parent; -1 for the root
    depth: np.ndarray     # int [m+1], 0 for the root
    node: np.ndarray      # int [m+1], node-table index (-1 for the root)
    mask: np.ndarray      # bool [m+1, m+1], mask[i, j] = row i may attend to row j

    def children(self, i: int) -> List[int]:
        return [j for j in range(len(self.token)) if self.parent[j] == i]

    def mask_words(self) -> np.ndarray:
        """Bit j of word j//64 of row i = mask[i, j] (uint64 [m+1, ceil((m+1)/64)])."""
        n = len(self.token)
        W = (n + 63) // 64
        out = np.zeros((n, W), dtype=np.uint64)
        for i in range(n):
            for j in range(n):
                if self.mask[i, j]:
                    out[i, j // 64] |= np.uint64(1) << np.uint64(j % 64)
        return out


def flatten(t: NodeTable, kept: Sequence[int], root_token: int) -> FlatTree:
    """The verify rows of a kept node set: the root at row 0, then the kept nodes in generation
    order (parents before children), each with its token, parent row, depth and ancestry mask
    (self, its ancestors and the root; EAGLE-2 page, "The Mask Preserves Tree Semantics in One
    Target Pass")."""
    order = sorted(kept)                      # generation order: parents precede children
    row_of = {node: r + 1 for r, node in enumerate(order)}
    n = len(order) + 1
    token = np.zeros(n, np.int64)
    parent = np.full(n, -1, np.int64)
    depth = np.zeros(n, np.int64)
    node = np.full(n, -1, np.int64)
    token[0] = root_token
    for r, i in enumerate(order, start=1):
        token[r] = t.token[i]
        p = t.parent[i]
        if p >= 0 and p not in row_of:
            raise ValueError("kept set is not ancestor-closed")
        parent[r] = 0 if p < 0 else row_of[p]
        depth[r] = t.depth[i]
        node[r] = i
    mask = np.zeros((n, n), dtype=bool)
    for r in range(n):
        a = r
        while a >= 0:
            mask[r, a] = True
            a = parent[a]
    return FlatTree(token, parent, depth, node, mask)


def grow_generic(children_of, depth: int, expand: int, budget: int) -> Tuple[NodeTable, List[int]]:
    """Expand-and-rerank with a callable drafter: children_of(path_tokens) -> [(token, conf)].
    Depth-1 nodes are the root's children; then `depth - 1` expansions of the best `expand`
    leaves; finally the global rerank keeps `budget` nodes. Returns (table, kept in rank order)."""
    t = NodeTable()
    for tok, c in children_of(()):
        t.add(tok, -1, np.log(F32(c), dtype=F32))
    for d in range(1, depth):
        for p in select_expand(t, d, expand):
            path = tuple(t.token[j] for j in t.path(p))
            for tok, c in children_of(path):
                t.add(tok, p, np.log(F32(c), dtype=F32))
    return t, rerank(t, budget)


def static_plan(parent: Sequence[int], rank: Sequence[int], k: int, depth: int):
    """Generation indices of a static topology's nodes and the k expansion rows per depth.

    parent[i] (-1 = child of the root, else an earlier node) and rank[i] (< k) describe
    node i. Returns (gen, rows): gen[i] = generation index of node i; rows[d] = the k
    generation indices expanded at depth d = 1 .. depth - 1. Generation indices follow
    the drafter's order: depth-1 nodes are 0..k-1 by rank; the children of the r-th row
    expanded at depth d start at k + (d - 1) k^2 + r k, in rank order."""
    n = len(parent)
    dep = [0] * n
    for i in range(n):
        if parent[i] >= i:
            raise ValueError("parents must precede their children")
        if not 0 <= rank[i] < k:
            raise ValueError("rank out of range")
        dep[i] = 1 if parent[i] < 0 else dep[parent[i]] + 1
        if dep[i] > depth:
            raise ValueError("node deeper than the draft depth")
    gen = [-1] * n
    for i in range(n):
        if dep[i] == 1:
            gen[i] = rank[i]
    rows = {}
    for d in range(1, depth):
        expanded = [i for i in range(n) if dep[i] == d and any(parent[j] == i for j in range(n))]
        if len(expanded) > k:
            raise ValueError("more than k nodes with children at one depth")
        row_gen = [gen[i] for i in expanded]
        lo = 0 if d == 1 else k + (d - 2) * k * k
        cnt = k if d == 1 else k * k
        for g in range(lo, lo + cnt):
            if len(row_gen) == k:
                break
            if g not in row_gen:
                row_gen.append(g)
        rows[d] = row_gen
        base = k + (d - 1) * k * k
        for r, i in enumerate(expanded):
            for j in range(n):
                if parent[j] == i:
                    gen[j] = base + r * k + rank[j]
    if len(set(gen)) != n:
        raise ValueError("two nodes share a parent and a rank")
    return gen, rows


def grow_static(children_of, parent: Sequence[int], rank: Sequence[int], k: int,
                depth: int) -> Tuple[NodeTable, List[int]]:
    """The static policy with a callable drafter (children_of as in grow_generic, returning
    at least k children): expand the planned rows, keep the topology's nodes."""
    gen, rows = static_plan(parent, rank, k, depth)
    t = NodeTable()
    for tok, c in children_of(())[:k]:
        t.add(tok, -1, np.log(F32(c), dtype=F32))
    for d in range(1, depth):
        for p in rows[d]:
            path = tuple(t.token[j] for j in t.path(p))
            for tok, c in children_of(path)[:k]:
                t.add(tok, p, np.log(F32(c), dtype=F32))
    return t, sorted(gen)


def chain_topology(depth: int):
    """A chain: one rank-0 child per depth."""
    return [i - 1 for i in range(depth)], [0] * depth


def is_ancestor_closed(t: NodeTable, kept: Sequence[int]) -> bool:
    """Every kept node's parent is kept or is the root (the closure the EAGLE lesson states for
    the top-m rerank)."""
    s = set(kept)
    return all(t.parent[i] < 0 or t.parent[i] in s for i in kept)
