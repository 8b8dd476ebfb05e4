"""Pins of the oracle's EAGLE-2 tree policy: the pages' hand-worked tree, the toy
builder's printed output, the ranking examples, and the ancestor-closure invariant."""
import itertools

import numpy as np
import pytest

from conftest import golden_lines
from oracle.tree import (NodeTable, chain_topology, flatten, grow_generic, grow_static, is_ancestor_closed,
                         rerank, select_expand, static_plan, topk_ids)


def _worked():
    conf, kept, values, expand2 = {}, [], {}, []
    for line in golden_lines("worked_tree.txt"):
        f = line.split()
        if f[0] == "conf":
            conf[f[1]] = float(f[2])
        elif f[0] == "kept":
            kept.append((f[1], float(f[2])))
        elif f[0] == "value":
            values[f[1]] = float(f[2])
        elif f[0] == "expand2":
            expand2 = f[1:]
    return conf, kept, values, expand2


def test_worked_example_tree():
    conf, kept, values, expand2 = _worked()
    letters = {}

    def children_of(path):
        name = "".join(letters[t] for t in path)
        out = []
        for key in sorted(conf):
            if len(key) == len(name) + 1 and key.startswith(name):
                tok = len(letters)
                letters.setdefault(tok, key[-1])
                out.append((tok, conf[key]))
        out.sort(key=lambda tc: -tc[1])
        return out

    t, ranked = grow_generic(children_of, depth=3, expand=2, budget=5)

    def name(i):
        return "".join(letters[t.token[j]] for j in t.path(i))

    # the two expanded depth-2 nodes are A->C and A->D (nothing under B)
    assert sorted(name(i) for i in select_expand(t, 2, 2)) == sorted(expand2)
    assert {name(i) for i in range(len(t))} == set(conf) - {"BEx"}
    assert [name(i) for i in ranked] == [k for k, _ in kept]
    for i in ranked:
        want = dict(kept)[name(i)]
        assert float(np.exp(t.logv[i])) == pytest.approx(want, rel=1e-6)
    for i in range(len(t)):
        if name(i) in values:
            assert float(np.exp(t.logv[i])) == pytest.approx(values[name(i)], rel=1e-6)
    assert is_ancestor_closed(t, ranked)
    # B->E has the larger own confidence but the smaller path value than A->D
    i_be = next(i for i in range(len(t)) if name(i) == "BE")
    i_ad = next(i for i in range(len(t)) if name(i) == "AD")
    assert conf["BE"] > conf["AD"] and t.logv[i_be] < t.logv[i_ad]


def _toy_cases():
    cases, paths = {}, {}
    for line in golden_lines("toy_dynamic_tree.txt"):
        f = line.split()
        if f[0] == "case":
            parts = line.split("|")
            head = parts[0].split()
            confs = [float(x) for x in head[2:5]]
            depths = [int(x) for x in parts[1].split()[1:]]
            total = float(parts[2].split()[1])
            cases[head[1]] = (confs, depths, total)
            paths[head[1]] = []
        elif f[0] == "path":
            paths[f[1]].append((tuple(int(x) for x in f[2].split(".")), float(f[3])))
    return cases, paths


def test_toy_builder_printed_output():
    cases, paths = _toy_cases()
    assert set(cases) == {"predictable", "uncertain"}
    for nm, (confs, depths, total) in cases.items():
        # tokens are the child ranks, so a node's token path is its rank path
        t, ranked = grow_generic(lambda path: list(enumerate(confs)), depth=3, expand=2, budget=6)
        got = [(tuple(t.token[j] for j in t.path(i)), round(float(np.exp(t.logv[i])), 3)) for i in ranked]
        assert got == paths[nm]
        assert sorted(t.depth[i] for i in ranked) == depths
        assert round(sum(float(np.exp(t.logv[i])) for i in ranked), 2) == total


def test_rank_examples():
    for line in golden_lines("rank_example.txt"):
        a1, c1, v1, a2, c2, v2 = [float(x) for x in line.split()[1:]]
        t = NodeTable()
        p1 = t.add(0, -1, np.log(np.float32(a1)))
        p2 = t.add(1, -1, np.log(np.float32(a2)))
        n1 = t.add(2, p1, np.log(np.float32(c1)))
        n2 = t.add(3, p2, np.log(np.float32(c2)))
        assert float(np.exp(t.logv[n1])) == pytest.approx(v1, rel=1e-6)
        assert float(np.exp(t.logv[n2])) == pytest.approx(v2, rel=1e-6)
        assert t.logv[n1] > t.logv[n2]


def _random_tree(rng, k, D, ties):
    t = NodeTable()
    pool = np.log(np.array([1.0, 0.5, 0.25, 0.125], np.float32))

    def logc():
        if ties:
            return pool[rng.integers(0, len(pool))]
        return np.float32(np.log(rng.uniform(1e-4, 1.0)))

    for j in range(k):
        t.add(j, -1, logc())
    for d in range(1, D):
        for p in select_expand(t, d, k):
            for j in range(k):
                t.add(j, p, logc())
    return t


@pytest.mark.parametrize("ties", [False, True])
def test_rerank_is_ancestor_closed(ties):
    """A confidence never exceeds 1, so a child's path value never exceeds its parent's;
    with ties broken toward shallower nodes the kept set is always a tree."""
    rng = np.random.default_rng(1 + ties)
    for _ in range(300):
        k, D = int(rng.integers(1, 5)), int(rng.integers(1, 6))
        t = _random_tree(rng, k, D, ties)
        for m in range(1, len(t) + 1):
            kept = rerank(t, m)
            assert is_ancestor_closed(t, kept)
            flatten(t, kept, 0)    # raises if not closed


def test_rerank_brute_force_small():
    """On tiny trees the rerank equals the best connected set by brute force:
    the m-subset maximising the sum of path values among ancestor-closed subsets
    (ties broken by the lexicographically smallest (depth, generation) list)."""
    rng = np.random.default_rng(5)
    for _ in range(40):
        t = _random_tree(rng, 2, 3, ties=False)
        for m in range(1, min(len(t), 6) + 1):
            best = None
            for sub in itertools.combinations(range(len(t)), m):
                if not is_ancestor_closed(t, sub):
                    continue
                score = sum(float(t.logv[i]) for i in sub)
                if best is None or score > best[0] + 1e-12:
                    best = (score, set(sub))
            # with distinct values the top-m set is also the max-sum closed set
            assert set(rerank(t, m)) == best[1]


def test_flatten_mask_semantics():
    rng = np.random.default_rng(2)
    for _ in range(50):
        t = _random_tree(rng, 3, 4, ties=False)
        kept = rerank(t, 9)
        ft = flatten(t, kept, 77)
        n = len(ft.token)
        assert ft.token[0] == 77 and ft.parent[0] == -1 and ft.depth[0] == 0
        for r in range(1, n):
            assert ft.parent[r] < r                              # parents precede children
            assert ft.depth[r] == ft.depth[ft.parent[r]] + 1
        for i in range(n):
            anc = set()
            a = i
            while a >= 0:
                anc.add(a)
                a = ft.parent[a]
            assert set(np.flatnonzero(ft.mask[i])) == anc       # root + ancestors + self
            assert ft.mask[i, 0]
        words = ft.mask_words()
        for i in range(n):
            for j in range(n):
                assert bool((int(words[i, j // 64]) >> (j % 64)) & 1) == ft.mask[i, j]


def test_chain_tree_mask_is_causal():
    t = NodeTable()
    p = -1
    for j in range(6):
        p = t.add(j, p, np.float32(-0.1))
    ft = flatten(t, rerank(t, 6), 9)
    assert np.array_equal(ft.mask, np.tril(np.ones((7, 7), dtype=bool)))


def test_topk_ids_ties_and_exclusion():
    v = np.array([1.0, 3.0, 3.0, 2.0, 3.0])
    assert list(topk_ids(v, 3)) == [1, 2, 4]
    assert list(topk_ids(v, 3, exclude=[2])) == [1, 4, 3]


# ---- static (EAGLE-1) trees ------------------------------------------------------------------
def _hash_drafter(vocab=50, k=4, seed=7):
    """Deterministic toy drafter: the children of a path are the k tokens with the largest
    pseudo-random score for (path, token), with those scores as confidences."""
    def children_of(path):
        rng = np.random.default_rng(abs(hash((seed,) + tuple(path))) % (2 ** 32))
        sc = rng.random(vocab)
        ids = sorted(range(vocab), key=lambda t: (-sc[t], t))[:k]
        tot = sum(sc[t] for t in ids) + 1.0
        return [(t, sc[t] / tot) for t in ids]
    return children_of


def test_static_chain_follows_the_top1_path():
    """A chain topology keeps exactly the drafter's greedy (rank-0) path."""
    children_of = _hash_drafter()
    for D in (1, 3, 5):
        parent, rank = chain_topology(D)
        t, kept = grow_static(children_of, parent, rank, k=4, depth=D)
        path, want = (), []
        for _ in range(D):
            tok = children_of(path)[0][0]
            want.append(tok)
            path = path + (tok,)
        got = [t.token[i] for i in kept]          # generation order = depth order for a chain
        assert got == want
        assert [t.depth[i] for i in kept] == list(range(1, D + 1))


def test_static_full_two_level_tree_equals_dynamic_keep_all():
    """Depth 2 with every depth-1 node expanded: the static policy keeps the same nodes as
    the dynamic one with the budget equal to all generated nodes."""
    k = 3
    children_of = _hash_drafter(k=k)
    parent = [-1] * k
    rank = list(range(k))
    for p in range(k):
        for r in range(k):
            parent.append(p)
            rank.append(r)
    ts, kept_s = grow_static(children_of, parent, rank, k=k, depth=2)
    td, kept_d = grow_generic(children_of, depth=2, expand=k, budget=k + k * k)
    assert ts.token == td.token and ts.parent == td.parent
    assert sorted(kept_s) == sorted(kept_d)


def test_static_kept_nodes_realise_the_topology():
    """Every kept node is its parent's rank-th child (children of a node in rank order), its
    depth is the topology's, and the kept set is ancestor-closed."""
    k, D = 3, 4
    children_of = _hash_drafter(k=k, seed=11)
    parent = [-1, -1, -1, 0, 0, 1, 3, 3, 5, 6]
    rank = [0, 1, 2, 0, 2, 1, 0, 1, 2, 0]
    gen, rows = static_plan(parent, rank, k, D)
    t, kept = grow_static(children_of, parent, rank, k=k, depth=D)
    assert kept == sorted(gen) and len(set(kept)) == len(parent)
    assert is_ancestor_closed(t, kept)
    for i, g in enumerate(gen):
        p = -1 if parent[i] < 0 else gen[parent[i]]
        assert t.parent[g] == p
        sib = [j for j in range(len(t)) if t.parent[j] == p]
        assert sib.index(g) == rank[i]
        a, dd = i, 0
        while a >= 0:
            a, dd = parent[a], dd + 1
        assert t.depth[g] == dd
    for d, r in rows.items():
        assert len(r) == k and len(set(r)) == k
        assert all(t.depth[g] == d for g in r)


def test_static_plan_rejects_bad_topologies():
    with pytest.raises(ValueError):
        static_plan([-1, 0], [0, 3], 3, 3)           # rank >= k
    with pytest.raises(ValueError):
        static_plan([-1, 0, 1, 2], [0, 0, 0, 0], 3, 3)  # deeper than D
    with pytest.raises(ValueError):
        static_plan([1, -1], [0, 0], 3, 3)            # parent after child
    with pytest.raises(ValueError):
        static_plan([-1, -1], [0, 0], 3, 3)           # same parent and rank twice
    with pytest.raises(ValueError, match="more than k"):   # three expanded depth-2 nodes, k = 2
        static_plan([-1, -1, 0, 0, 1, 2, 3, 4], [0, 1, 0, 1, 0, 0, 0, 0], 2, 3)
