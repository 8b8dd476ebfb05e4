"""Pins of the oracle's drafter wiring by constructed weights (see wiring_weights.py).

What the pages fix, and what each test checks against a value computed here from the
target alone (never from the oracle's drafter code):

- EAGLE-1 drafter position p reads the target feature f_p, the LM head's input
  ("EAGLE: Feature-Level Drafting", "The big idea: draft at the feature level";
  "EAGLE 三代" §2.1): with the drafter reduced to the identity on its feature input,
  the root's candidates after prefill are the top-k of the target's logits at the last
  prompt position, and after a cycle the top-k of its logits at the last accepted row.
- EAGLE-1 drafter position p reads the token one step ahead, x_{p+1} ("Resolving the
  uncertainty by feeding back the token"): with the identity on the token input, the
  candidates are the top-k of the LM head applied to the embedding of the first
  generated token, and after a cycle to that of the bonus token.
- EAGLE-3 fuses the residual-stream outputs of target layers l, m, h (0-based) and,
  below the root, feeds the drafter its parent's output a in place of g ("EAGLE 三代"
  §4.3): with the fusion FC keeping one block and the attention output zeroed, the root
  row's output is Phi(g) = x + MLP(x) at x = g, the children of a depth-d node are the
  top-k of the LM head at Phi^(d+1)(g), and after a cycle the root's candidates come
  from the g of the last accepted row.

Each test also checks that the rival readings (f of the next position, the pre-norm
residual, the unshifted token, another capture layer, g in place of a) would give other
candidates, so the pin can fail."""
import dataclasses

import numpy as np
import pytest

from eagle_speculative_decoding_cycle_gb300 import synth
from oracle.cycle import OracleSeq, build_model
from oracle.model import KV, quantizer, rmsnorm
from wiring_weights import constructed, eagle3_workload, f32_model

K_TOL = 1e-6


def _topk(logits, k):
    """k largest, ties to the lower id (the pages' argmax with the lowest-id reading)."""
    order = np.lexsort((np.arange(logits.shape[0]), -logits))
    return [int(i) for i in order[:k]]


def _logc(logits, ids):
    mx = np.max(logits)
    lse = mx + np.log(np.sum(np.exp(logits - mx)))
    return np.array([logits[i] - lse for i in ids])


def _forward(M, wl, tokens, n_layers=None, final=True):
    """Causal forward of the target over `tokens` run layer by layer here: the residual
    stream after `n_layers` layers, or the final-norm output (the LM head's input)."""
    s = wl.model
    q = quantizer(s.dtype)
    tokens = np.asarray(tokens)
    n = len(tokens)
    kv = KV.empty(s.n_layers, s.n_kv_heads, n, s.head_dim, s.dtype)
    pos = np.arange(n)
    vis = np.tril(np.ones((n, n), dtype=bool))
    x = np.asarray(M.W["embed"][tokens], np.float64)
    for li in range(s.n_layers if n_layers is None else n_layers):
        L = M.layers[li]
        x = M.layer_rows(L, x, q(rmsnorm(x, L.attn_norm, s.rms_eps)), pos, kv, li, pos, vis)
    if final:
        return q(rmsnorm(x, M.W["final_norm"], s.rms_eps))
    return x


def _lm(M, f):
    return np.asarray(f, np.float64) @ np.asarray(M.W["lm_head"], np.float64).T


def _phi(M, wl, x):
    """x + MLP(x) with the drafter layer's MLP, rounded at the model's rounding points
    (the SwiGLU MLP of a Llama-style layer, restated here)."""
    s = wl.model
    q = quantizer(s.dtype)
    W = M.W
    F = s.ffn
    x = np.asarray(x, np.float64)
    n2 = q(x / np.sqrt(np.mean(x * x) + s.rms_eps) * np.asarray(W["draft.mlp_norm"], np.float64))
    wgu = np.asarray(W["draft.wgu"], np.float64)
    gate, up = wgu[:F] @ n2, wgu[F:] @ n2
    h = q(gate / (1.0 + np.exp(-gate)) * up)
    return q(x + np.asarray(W["draft.wd"], np.float64) @ h)


def _setup(wl, select):
    W = synth.weights_to_numpy(constructed(wl, select))
    M = build_model(W, wl)
    prompt = synth.make_prompts(wl)[0].numpy()
    o = OracleSeq(M, wl)
    return M, prompt, o


def _check_cands(o, logits, k):
    ids = _topk(logits, k)
    assert o.cand_tok == ids
    assert np.allclose(np.asarray(o.cand_logc, np.float64), _logc(logits, ids), atol=K_TOL, rtol=0)


WL1 = synth.TINY.replace(tree=synth.TreeShape(topk=4, depth=3, m=10))


def test_eagle1_drafter_reads_the_lm_head_input_of_its_own_position():
    wl = WL1
    M, prompt, o = _setup(wl, "feature")
    k = wl.tree.topk
    first = o.prefill(prompt)
    f = _forward(M, wl, prompt)
    want = _lm(M, f[-1])
    _check_cands(o, want, k)
    assert first == _topk(want, 1)[0]
    # rival readings give other candidates: the pre-norm residual (other confidences) and
    # the feature of the next position (the first generated token's row)
    pre = _lm(M, _forward(M, wl, prompt, final=False)[-1])
    assert not np.allclose(_logc(pre, _topk(pre, k)), _logc(want, _topk(want, k)), atol=1e-3)
    nxt = _lm(M, _forward(M, wl, list(prompt) + [first])[-1])
    assert _topk(nxt, k) != _topk(want, k)
    for _ in range(3):
        o.cycle()
        seq = list(prompt) + o.committed[:-1]
        want = _lm(M, _forward(M, wl, seq)[-1])
        _check_cands(o, want, k)
        assert o.cand_tok[0] == o.committed[-1]      # greedy: the bonus is that row's argmax


def test_eagle1_drafter_reads_the_token_one_step_ahead():
    wl = WL1
    M, prompt, o = _setup(wl, "token")
    k = wl.tree.topk
    first = o.prefill(prompt)
    E = np.asarray(M.W["embed"], np.float64)
    _check_cands(o, _lm(M, E[first]), k)
    assert _topk(_lm(M, E[prompt[-1]]), k) != _topk(_lm(M, E[first]), k)   # unshifted token
    for _ in range(3):
        o.cycle()
        _check_cands(o, _lm(M, E[o.committed[-1]]), k)


_E3 = f32_model(synth.SMALL_BF16_E3)
WL3 = eagle3_workload(_E3.replace(model=dataclasses.replace(_E3.model, n_layers=4),
                                  tree=synth.TreeShape(topk=3, depth=4, m=9)), fuse=(0, 1, 2))


@pytest.mark.parametrize("select", [0, 1, 2], ids=["l", "m", "h"])
def test_eagle3_fuses_residual_outputs_and_substitutes_a(select):
    wl = WL3
    M, prompt, o = _setup(wl, select)
    k, D = wl.tree.topk, wl.tree.depth
    layer = wl.drafter.fuse_layers[select]
    o.prefill(prompt)
    g = _forward(M, wl, prompt, n_layers=layer + 1, final=False)[-1]
    g = quantizer(wl.model.dtype)(g)
    a = _phi(M, wl, g)
    _check_cands(o, _lm(M, a), k)
    # rival capture reading: the residual before the layer
    before = quantizer(wl.model.dtype)(_forward(M, wl, prompt, n_layers=layer, final=False)[-1])
    assert _topk(_lm(M, _phi(M, wl, before)), k) != _topk(_lm(M, a), k)
    # below the root every drafter row takes its parent's output: the children of a
    # depth-d node are the top-k at Phi^(d+1)(g)
    plan = o.draft_and_verify()
    t = plan.table
    chain = [a]
    for d in range(1, D):
        chain.append(_phi(M, wl, chain[-1]))
    for v in range(len(t.token)):
        kids = [i for i in range(len(t.token)) if t.parent[i] == v]
        if kids:
            d = t.depth[v]
            want = _lm(M, chain[d])
            assert [t.token[i] for i in kids] == _topk(want, k)
            assert np.allclose([float(t.logv[i]) - float(t.logv[v]) for i in kids],
                               _logc(want, _topk(want, k)), atol=1e-4)
    assert _topk(_lm(M, chain[1]), k) != _topk(_lm(M, chain[0]), k)   # g in place of a differs
    path, bonus = o.decide(plan)
    o.commit(plan, path, bonus)
    seq = list(prompt) + o.committed[:-1]
    g_last = quantizer(wl.model.dtype)(_forward(M, wl, seq, n_layers=layer + 1, final=False)[-1])
    _check_cands(o, _lm(M, _phi(M, wl, g_last)), k)
