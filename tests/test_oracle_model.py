"""Pins of the oracle's layer math against independent library formulations (torch
fp64 CPU ops), and of the tree-attention semantics: a tree row must equal plain
causal decoding of its own root-to-node path."""
import dataclasses

import numpy as np
import pytest
import torch
import torch.nn.functional as Fn

from eagle_speculative_decoding_cycle_gb300 import synth
from oracle.cycle import OracleSeq, build_model
from oracle.model import KV, attention, rmsnorm, rope, silu
from oracle.tree import NodeTable, flatten, rerank, select_expand


def test_rmsnorm_matches_torch():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((7, 33)) * 3
    g = rng.standard_normal(33)
    want = Fn.rms_norm(torch.from_numpy(x), (33,), torch.from_numpy(g), eps=1e-5).numpy()
    assert np.allclose(rmsnorm(x, g, 1e-5), want, rtol=1e-13, atol=1e-13)


def test_rope_matches_complex_rotation():
    """Rotate-half RoPE equals multiplying (x_i + i x_{i+d/2}) by exp(i pos theta^(-2i/d))."""
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, 3, 16))
    pos = np.array([0, 1, 7, 100, 4095])
    z = x[..., :8] + 1j * x[..., 8:]
    ang = pos[:, None] * (1e4 ** (-np.arange(8) * 2.0 / 16))[None, :]
    zr = z * np.exp(1j * ang)[:, None, :]
    want = np.concatenate([zr.real, zr.imag], axis=-1)
    assert np.allclose(rope(x, pos, 1e4), want, rtol=1e-12, atol=1e-12)


def test_silu_matches_torch():
    x = np.linspace(-20, 20, 1001)
    assert np.allclose(silu(x), Fn.silu(torch.from_numpy(x)).numpy(), rtol=1e-14, atol=1e-15)


@pytest.mark.parametrize("nq,nkv", [(4, 4), (8, 2)])
def test_attention_causal_matches_sdpa(nq, nkv):
    """A chain tree's mask is the causal mask: the oracle attention with it equals
    torch's scaled_dot_product_attention (is_causal, GQA by head repetition)."""
    rng = np.random.default_rng(2)
    S, d = 13, 16
    q = rng.standard_normal((S, nq, d))
    K = rng.standard_normal((nkv, S, d))
    V = rng.standard_normal((nkv, S, d))
    got = attention(q, K, V, np.tril(np.ones((S, S), dtype=bool)))
    qt = torch.from_numpy(q).permute(1, 0, 2)[None]
    kt = torch.from_numpy(np.repeat(K, nq // nkv, axis=0))[None]
    vt = torch.from_numpy(np.repeat(V, nq // nkv, axis=0))[None]
    want = Fn.scaled_dot_product_attention(qt, kt, vt, is_causal=True)[0].permute(1, 0, 2).numpy()
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)


def _f64(wl):
    return wl.replace(model=dataclasses.replace(wl.model, dtype="f64"))


@pytest.mark.parametrize("base", [synth.TINY, synth.SMALL_BF16_E3])
def test_tree_rows_equal_plain_path_decoding(base):
    """Each flattened row of a verify pass sees ctx + root + its ancestors only, so its
    feature equals a plain causal forward of the sequence ctx, root, ancestors, node."""
    wl = _f64(base)
    W = synth.weights_to_numpy(synth.make_weights(wl))
    M = build_model(W, wl)
    s = wl.model
    rng = np.random.default_rng(3)
    n = 9
    ctx = rng.integers(0, s.vocab, n)
    t = NodeTable()
    for j in range(3):
        t.add(int(rng.integers(0, s.vocab)), -1, np.float32(np.log(rng.uniform(0.05, 1))))
    for d in range(1, 3):
        for p in select_expand(t, d, 2):
            for j in range(3):
                t.add(int(rng.integers(0, s.vocab)), p, np.float32(np.log(rng.uniform(0.05, 1))))
    ft = flatten(t, rerank(t, 8), int(rng.integers(0, s.vocab)))
    kv = KV.empty(s.n_layers, s.n_kv_heads, 64, s.head_dim, "f64")
    pos = np.arange(n)
    M.target_rows(ctx, pos, kv, pos, np.tril(np.ones((n, n), dtype=bool)))
    rows = len(ft.token)
    vis = np.zeros((rows, n + rows), dtype=bool)
    vis[:, :n] = True
    vis[:, n:] = ft.mask
    f_tree, _ = M.target_rows(ft.token, n + ft.depth, kv, n + np.arange(rows), vis)
    for r in range(rows):
        chain = [r]
        while ft.parent[chain[-1]] >= 0:
            chain.append(ft.parent[chain[-1]])
        seq = np.concatenate([ctx, ft.token[chain[::-1]]])
        kv2 = KV.empty(s.n_layers, s.n_kv_heads, 64, s.head_dim, "f64")
        L = len(seq)
        p2 = np.arange(L)
        f_plain, _ = M.target_rows(seq, p2, kv2, p2, np.tril(np.ones((L, L), dtype=bool)))
        assert np.allclose(f_tree[r], f_plain[-1], rtol=1e-11, atol=1e-11)


def test_drafter_tree_rows_equal_causal_drafter_chain():
    """The drafter's expansion rows attend to the drafter context plus their expanded
    ancestors: a depth-d row's output equals running the drafter causally over the
    context followed by the chain of (parent feature, token) rows of its path."""
    wl = _f64(synth.TINY.replace(tree=synth.TreeShape(topk=3, depth=4, m=10)))
    W = synth.weights_to_numpy(synth.make_weights(wl))
    M = build_model(W, wl)
    prompt = synth.make_prompts(wl)[0].numpy()[:12]
    o = OracleSeq(M, wl)
    o.prefill(prompt)
    plan = o.draft_and_verify()
    t = plan.table
    # re-derive one deepest expanded path and replay it causally
    deep = [i for i in range(len(t)) if t.depth[i] == wl.tree.depth]
    v = deep[0]
    chain = t.path(v)[:-1]              # expanded ancestors, depth 1 .. D-1
    o2 = OracleSeq(M, wl)
    o2.prefill(prompt)
    n = o2.n
    feats, toks = [o2.root_feat], []
    out = None
    for j, a in enumerate(chain):
        toks.append(t.token[a])
        P = n + j + 1
        pos = np.arange(n, P)
        vis = np.zeros((len(pos), P), dtype=bool)
        for r in range(len(pos)):
            vis[r, :n + r + 1] = True
        dkv = KV(o2.dkv.k.copy(), o2.dkv.v.copy())
        out = M.drafter_rows(np.stack(feats), np.array(toks), pos, dkv, pos, vis)
        feats.append(out[-1])
    # the deepest expanded ancestor's children came from its drafter output
    ids, lcs = o2._candidates(out[-1], -1, 0, len(chain) + 1)
    kids = [i for i in range(len(t)) if t.parent[i] == chain[-1]]
    assert [t.token[i] for i in kids] == ids
    assert np.allclose([float(t.logv[i]) - float(t.logv[chain[-1]]) for i in kids], lcs, atol=1e-5)
