"""Pins of the oracle's EAGLE-3 training-time-test forward.

- Step 1 is the plain causal drafter pass over the sequence (the drafter's prefill).
- The step-s row of source t equals what inference computes when it drafts s - 1 more
  steps after a context ending at t, feeding each step's output a back in place of g with
  the given tokens: the chain rebuilt row by row in contiguous slots after the context.
- The loss is the mean cross-entropy, checked against scipy's log-softmax."""
import dataclasses

import numpy as np
import pytest
from scipy.special import log_softmax

from eagle_speculative_decoding_cycle_gb300 import synth
from oracle.cycle import build_model
from oracle.model import KV
from oracle.ttt import cross_entropy, ttt_forward

N, STEPS = 12, 3


def _model(wl):
    return build_model(synth.weights_to_numpy(synth.make_weights(wl)), wl)


def _seq(wl, n=N, seed=5):
    return np.random.default_rng(seed).integers(0, wl.model.vocab, n)


def _features(M, x):
    n = len(x)
    s = M.s
    kv = KV.empty(s.n_layers, s.n_kv_heads, n, s.head_dim, s.dtype)
    pos = np.arange(n)
    f, caps = M.target_rows(x, pos, kv, pos, np.tril(np.ones((n, n), dtype=bool)))
    return f if M.drafter_kind == 1 else M.fuse(caps)


WORKLOADS = [synth.SMALL_BF16_E3, synth.TINY]


@pytest.mark.parametrize("wl", WORKLOADS, ids=lambda w: w.name)
def test_step1_is_the_causal_drafter_pass(wl):
    M = _model(wl)
    x = _seq(wl)
    g = _features(M, x)
    s = M.s
    dkv = KV.empty(1, s.n_kv_heads, N, s.head_dim, s.dtype)
    rows = np.arange(N - 1)
    want = M.drafter_rows(g[rows], x[rows + 1], rows, dkv, rows, np.tril(np.ones((N - 1, N), dtype=bool)))
    _, outs = ttt_forward(M, x, STEPS)
    np.testing.assert_array_equal(outs[0], want[:N - 2])


@pytest.mark.parametrize("wl", WORKLOADS, ids=lambda w: w.name)
def test_later_steps_equal_inference_drafting(wl):
    M = _model(wl)
    x = _seq(wl)
    g = _features(M, x)
    _, outs = ttt_forward(M, x, STEPS)
    s_ = M.s
    for t in (0, 3, N - 2 - STEPS):
        # inference: the drafter's causal context 0..t, then one row per further step in the
        # next contiguous slots, each seeing the context and the chain so far
        dkv = KV.empty(1, s_.n_kv_heads, N + STEPS, s_.head_dim, s_.dtype)
        ctx = np.arange(t + 1)
        vis = np.zeros((t + 1, N + STEPS), dtype=bool)
        vis[:, :t + 1] = np.tril(np.ones((t + 1, t + 1), dtype=bool))
        a = M.drafter_rows(g[ctx], x[ctx + 1], ctx, dkv, ctx, vis)[-1:]
        np.testing.assert_array_equal(a, outs[0][t:t + 1])
        for j in range(2, STEPS + 1):
            slot = t + j - 1
            v = np.zeros((1, N + STEPS), dtype=bool)
            v[0, :slot + 1] = True
            a = M.drafter_rows(a, x[[t + j]], np.array([t + j - 1]), dkv, np.array([slot]), v)
            np.testing.assert_allclose(a, outs[j - 1][t:t + 1], rtol=0, atol=1e-6)


def test_cross_entropy_is_minus_log_softmax():
    rng = np.random.default_rng(0)
    for _ in range(5):
        z = rng.normal(size=37) * 3
        t = int(rng.integers(0, 37))
        assert cross_entropy(z, t) == pytest.approx(-log_softmax(z)[t], rel=1e-12, abs=1e-12)


def test_step_losses_are_mean_cross_entropies():
    wl = synth.SMALL_BF16_E3
    M = _model(wl)
    x = _seq(wl)
    losses, outs = ttt_forward(M, x, STEPS)
    for s, (loss, a) in enumerate(zip(losses, outs), start=1):
        lg = M.logits(a)
        want = np.mean([-log_softmax(lg[t])[x[t + s + 1]] for t in range(len(a))])
        assert loss == pytest.approx(want, rel=1e-10)
    with pytest.raises(ValueError):
        ttt_forward(M, x[:STEPS + 2], STEPS)
