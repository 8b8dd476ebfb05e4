"""Pins of the oracle's EAGLE-2 tree policy: the pages' hand-worked tree, the toy
builder's printed output, the ranking examples, and the ancestor-closure invariant."""
import itertools

import numpy as np
import pytest

from conftest import golden_lines
from oracle.tree import (NodeTable, flatten, grow_generic, is_ancestor_closed, rerank,
                         select_expand, topk_ids)


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
