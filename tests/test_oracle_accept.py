"""Pins of the oracle's acceptance rule and KV compaction: greedy speculative output
equals plain greedy decoding; the exact outcome distribution of the sampling rule,
enumerated branch by branch on a vocabulary-16 model, equals the target's own
autoregressive joint; the sampled walk follows that distribution; compaction leaves
the KV cache that plain decoding would have built."""
import dataclasses
from collections import defaultdict

import numpy as np
import pytest
from scipy import stats

from eagle_speculative_decoding_cycle_gb300 import synth
from oracle import philox
from oracle.accept import compact, enumerate_walk, sample_walk
from oracle.cycle import OracleSeq, build_model, plain_decode
from oracle.model import KV, logsumexp
from oracle.speedup import expected_tokens
from oracle.tree import NodeTable, flatten, rerank


def _setup(wl):
    W = synth.weights_to_numpy(synth.make_weights(wl))
    return build_model(W, wl), synth.make_prompts(wl)[0].numpy()


@pytest.mark.parametrize("wl,planted", [(synth.TINY, True), (synth.TINY, False),
                                        (synth.SMALL_BF16, True),
                                        (synth.SMALL_BF16_E3.replace(
                                            tree=dataclasses.replace(synth.SMALL_BF16_E3.tree, temperature=0.0)),
                                         True)])
def test_greedy_speculative_equals_plain(wl, planted):
    M, prompt = _setup(wl)
    N = wl.new_tokens
    R = plain_decode(M, wl, prompt, N + wl.tree.depth + 2)
    o = OracleSeq(M, wl)
    o.prefill(prompt, R if planted else None)
    assert o.generate(N) == R[:N]
    if planted:
        assert max(o.accept_lengths) >= 2          # deep paths were exercised


# static trees for the tiny model (k = 4, D = 4): a chain, and an m = 16 two-branch shape
_TINY_CHAIN = synth.TINY.replace(tree=dataclasses.replace(synth.TINY.tree, m=4, static_parent=(-1, 0, 1, 2),
                                                         static_rank=(0, 0, 0, 0)))
_TINY_STATIC = synth.TINY.replace(tree=dataclasses.replace(
    synth.TINY.tree, m=16,
    static_parent=(-1, -1, -1, 0, 0, 0, 1, 1, 2, 3, 3, 4, 6, 9, 9, 10),
    static_rank=(0, 1, 2, 0, 1, 2, 0, 1, 0, 0, 1, 0, 0, 0, 1, 0)))


@pytest.mark.parametrize("wl", [_TINY_CHAIN, _TINY_STATIC])
def test_greedy_speculative_equals_plain_static_tree(wl):
    """The static (EAGLE-1) tree keeps the output lossless and verifies exactly its shape."""
    M, prompt = _setup(wl)
    N = wl.new_tokens
    R = plain_decode(M, wl, prompt, N + wl.tree.depth + 2)
    o = OracleSeq(M, wl)
    o.prefill(prompt, R)
    assert o.generate(N) == R[:N]
    assert max(o.accept_lengths) >= 2


def _f64(wl):
    return wl.replace(model=dataclasses.replace(wl.model, dtype="f64"))


def test_sampling_rule_exact_joint_vocab16():
    """Enumerate every accept/reject/bonus branch over as many cycles as needed to
    commit 3 tokens after the prefill token; the joint must equal the product of the
    target's conditionals p(t1|x) p(t2|x,t1) p(t3|x,t1,t2) to 1e-12."""
    wl = _f64(synth.VOCAB16)
    M, prompt = _setup(wl)
    T = wl.tree.temperature
    need = 3
    o = OracleSeq(M, wl)
    first = o.prefill(prompt)
    stats_ = {"plans": 0, "accepts": 0}

    def spec_joint(o, need):
        plan = o.draft_and_verify()
        stats_["plans"] += 1
        res = defaultdict(float)
        for path, bonus, prob in o.outcomes(plan):
            toks = [int(plan.flat.token[r]) for r in path] + [bonus]
            stats_["accepts"] += len(path) > 0
            if len(toks) >= need:
                res[tuple(toks[:need])] += prob
            else:
                o2 = o.fork()
                o2.commit(plan, path, bonus)
                for k2, p2 in spec_joint(o2, need - len(toks)).items():
                    res[tuple(toks) + k2] += prob * p2
        return res

    got = spec_joint(o, need)
    V = wl.model.vocab
    s = wl.model

    def cond(seq):
        kv = KV.empty(s.n_layers, s.n_kv_heads, len(seq) + 1, s.head_dim, "f64")
        L = len(seq)
        pos = np.arange(L)
        f, _ = M.target_rows(np.asarray(seq), pos, kv, pos, np.tril(np.ones((L, L), dtype=bool)))
        lg = M.logits(f[-1:])[0] / T
        return np.exp(lg - logsumexp(lg))

    base = list(prompt) + [first]
    p1 = cond(base)
    total = 0.0
    for a in range(V):
        p2 = cond(base + [a])
        for b in range(V):
            p3 = cond(base + [a, b])
            for c in range(V):
                want = p1[a] * p2[b] * p3[c]
                assert abs(got.get((a, b, c), 0.0) - want) < 1e-12
                total += got.get((a, b, c), 0.0)
    assert abs(total - 1.0) < 1e-12
    assert stats_["accepts"] > 0 and stats_["plans"] > 1   # both branches were exercised


def test_enumerate_walk_marginals_single_node():
    rng = np.random.default_rng(4)
    for _ in range(50):
        V = 12
        p = rng.dirichlet(np.ones(V) * 0.5)
        kids = list(rng.choice(V, size=int(rng.integers(0, 5)), replace=False))
        t = NodeTable()
        for k in kids:
            t.add(int(k), -1, np.float32(-1.0))
        ft = flatten(t, list(range(len(kids))), 0)
        probs = np.tile(p, (len(ft.token), 1))
        marg = np.zeros(V)
        for path, bonus, prob in enumerate_walk(ft, probs):
            first = int(ft.token[path[0]]) if path else bonus
            marg[first] += prob
        assert np.allclose(marg, p, atol=1e-14)


def test_sampled_walk_follows_enumerated_distribution():
    """The Philox-driven walk (fp32 threshold test, Gumbel-argmax bonus) against the
    exact outcome probabilities of a fixed two-level tree: chi-square at p > 0.001."""
    rng = np.random.default_rng(6)
    V = 8
    probs = rng.dirichlet(np.ones(V), size=4)
    t = NodeTable()
    a = t.add(int(np.argmax(probs[0])), -1, np.float32(-0.1))
    t.add(int(np.argsort(probs[0])[-2]), -1, np.float32(-0.5))
    t.add(3, a, np.float32(-0.2))
    ft = flatten(t, [0, 1, 2], 0)
    exact = defaultdict(float)
    for path, bonus, prob in enumerate_walk(ft, probs):
        exact[(tuple(path), bonus)] += prob
    N = 40000
    counts = defaultdict(int)
    logp = np.log(probs)
    for trial in range(N):
        def uni(row, i):
            return philox.draw_uniform(9, philox.STREAM_ACCEPT, 0, trial, i, row)

        def bonus(row, excl):
            g = philox.gumbel_row(9, philox.STREAM_GUMBEL, 0, trial, row, V)
            v = logp[row] + g
            v[np.asarray(excl, dtype=np.int64)] = -np.inf
            return int(np.argmax(v))

        path, b = sample_walk(ft, lambda r, tok: probs[r][tok], uni, bonus)
        counts[(tuple(path), b)] += 1
    keys = sorted(exact)
    obs = np.array([counts[k] for k in keys], dtype=np.float64)
    exp = np.array([exact[k] for k in keys]) * N
    assert sum(counts[k] for k in counts if k not in exact) == 0
    big = exp >= 5
    o = np.append(obs[big], obs[~big].sum())
    e = np.append(exp[big], exp[~big].sum())
    if e[-1] < 5:
        o[-2] += o[-1]; e[-2] += e[-1]
        o, e = o[:-1], e[:-1]
    assert stats.chisquare(o, e).pvalue > 1e-3


def test_compact_is_read_all_then_write():
    rng = np.random.default_rng(7)
    k = rng.standard_normal((2, 3, 20, 4))
    v = rng.standard_normal((2, 3, 20, 4))
    k0, v0 = k.copy(), v.copy()
    n, path = 5, [2, 5, 9]           # slot n+2 is both a source and a target
    compact(k, v, n, path)
    for j, r in enumerate(path, start=1):
        assert np.array_equal(k[:, :, n + j], k0[:, :, n + r])
        assert np.array_equal(v[:, :, n + j], v0[:, :, n + r])
    assert np.array_equal(k[:, :, :n + 1], k0[:, :, :n + 1])


def test_compacted_cache_equals_plain_decode_cache():
    wl = _f64(synth.TINY)
    M, prompt = _setup(wl)
    R = plain_decode(M, wl, prompt, 40)
    o = OracleSeq(M, wl)
    o.prefill(prompt, R)
    while len(o.committed) < 30:
        o.cycle()
    toks = list(prompt) + o.committed[:-1]       # everything but the root is cached
    s = wl.model
    L = len(toks)
    assert L == o.n
    kv = KV.empty(s.n_layers, s.n_kv_heads, L, s.head_dim, "f64")
    pos = np.arange(L)
    M.target_rows(np.asarray(toks), pos, kv, pos, np.tril(np.ones((L, L), dtype=bool)))
    assert np.allclose(o.kv.k[:, :, :L], kv.k, rtol=1e-11, atol=1e-11)
    assert np.allclose(o.kv.v[:, :, :L], kv.v, rtol=1e-11, atol=1e-11)
    assert max(o.accept_lengths) >= 2


def test_planted_tau_matches_closed_form():
    """Planted mode: tau per cycle = 1 + run of planted depths, E[tau] = sum_{i<=D} p^i."""
    taus = []
    for seed in range(6):
        wl = synth.TINY.replace(seed=seed)
        M, prompt = _setup(wl)
        R = plain_decode(M, wl, prompt, wl.new_tokens + wl.tree.depth + 2)
        o = OracleSeq(M, wl)
        o.prefill(prompt, R)
        o.generate(wl.new_tokens)
        taus += [L + 1 for L in o.accept_lengths]
    taus = np.array(taus, dtype=np.float64)
    want = expected_tokens(wl.tree.planted_p, wl.tree.depth)
    se = taus.std() / np.sqrt(len(taus))
    assert abs(taus.mean() - want) < 4 * se + 0.05
