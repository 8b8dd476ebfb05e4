"""Parity at the full Llama-2-7B shape (H 4096, vocab 32000, k10 D6 m60), in the launch
configuration the bench uses, on sampled outputs the oracle can compute: the GPU verify
logits of the rows along the deepest kept tree path against the oracle's plain causal
forward of that path (each tree row sees only its own ancestors).

Tolerance. At two layers of the full-width model the logits must agree within the bf16
bound 5e-2. Over the full 32 layers the rounding noise of any fp32-accumulating
implementation exceeds that bound on this random-init model: bf16 rounding points sit
after every projection, fp32 sums land on the other side of a rounding boundary a few
times per row and layer, and those one-ulp differences accumulate with depth. The
full-depth check therefore measures that floor on the same rows -- the oracle with its
matmuls accumulated in fp32 against the oracle in fp64 -- and requires the GPU's
deviation to stay within twice it (max-abs and rms)."""
import dataclasses

import numpy as np
import pytest
import torch

from eagle_speculative_decoding_cycle_gb300 import _lib as L
from eagle_speculative_decoding_cycle_gb300 import api, synth
from oracle import model as om
from oracle.cycle import build_model
from oracle.model import KV
from oracle.tree import NodeTable, flatten, rerank

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.fixture(scope="module")
def weights():
    w = synth.make_weights(synth.LLAMA2_7B.replace(prompt_len=(16, 16)), device=DEV)
    yield w
    del w
    torch.cuda.empty_cache()


def gpu_chain(wl, weights, prompt):
    """One GPU cycle; returns (verify logits of the deepest path's rows, path tokens)."""
    eng = api.Engine(wl, weights, max_ctx=256)
    eng.prefill([prompt.to(DEV)])
    eng.set_debug(L.DEBUG_LOGITS)
    eng.cycle()
    eng.sync()
    gl = eng.dump(L.DUMP_VERIFY_LOGITS).double().numpy()
    tok, pos, par, node, mask = eng.dump(L.DUMP_TREE)
    tok, par = tok[0].tolist(), par[0].tolist()
    ntok, npar, ndep, nlogv = eng.dump(L.DUMP_NODES)
    t = NodeTable(ntok[0].tolist(), npar[0].tolist(), ndep[0].tolist(), [np.float32(x) for x in nlogv[0].numpy()])
    ft = flatten(t, rerank(t, wl.tree.m), tok[0])
    assert ft.token.tolist() == tok and ft.parent.tolist() == par
    chain = [int(np.argmax(ft.depth))]
    while par[chain[-1]] >= 0:
        chain.append(par[chain[-1]])
    chain = chain[::-1]
    eng.close()
    return gl[chain], [tok[r] for r in chain]


def oracle_chain(wl, weights, prompt, chain_tokens, fp32_matmul=False):
    keep = ["embed", "lm_head", "final_norm"] + [k for k in weights if k.startswith("layers.")]
    Wn = {k: weights[k].to("cpu", torch.float32).numpy() for k in keep}
    M = build_model(Wn, wl.replace(drafter=synth.DrafterShape(kind=1)))
    seq = prompt.tolist() + chain_tokens
    n = len(seq)
    s = wl.model
    kv = KV.empty(s.n_layers, s.n_kv_heads, n, s.head_dim)
    p = np.arange(n)
    orig = om.mm
    if fp32_matmul:
        om.mm = lambda a, w: (np.asarray(a, np.float32) @ np.asarray(w, np.float32).T).astype(np.float64)
    try:
        f, _ = M.target_rows(np.asarray(seq), p, kv, p, np.tril(np.ones((n, n), dtype=bool)))
        return M.logits(f[-len(chain_tokens):])
    finally:
        om.mm = orig


def _truncate(weights, n_layers):
    return {k: v for k, v in weights.items() if not k.startswith("layers.") or int(k.split(".")[1]) < n_layers}


def test_full_width_two_layers_within_bf16_tolerance(weights):
    base = synth.LLAMA2_7B.replace(prompt_len=(16, 16))
    wl = base.replace(model=dataclasses.replace(base.model, n_layers=2))
    w = _truncate(weights, 2)
    prompt = synth.make_prompts(base)[0]
    gl, toks = gpu_chain(wl, w, prompt)
    want = oracle_chain(wl, w, prompt, toks)
    assert np.max(np.abs(gl - want)) < 5e-2


def test_full_depth_within_fp32_accumulation_floor(weights):
    wl = synth.LLAMA2_7B.replace(prompt_len=(16, 16))
    prompt = synth.make_prompts(wl)[0]
    gl, toks = gpu_chain(wl, weights, prompt)
    want = oracle_chain(wl, weights, prompt, toks)
    floor = np.abs(oracle_chain(wl, weights, prompt, toks, fp32_matmul=True) - want)
    err = np.abs(gl - want)
    print(f"full depth: GPU max {err.max():.4f} rms {np.sqrt((err ** 2).mean()):.4f}; "
          f"fp32 floor max {floor.max():.4f} rms {np.sqrt((floor ** 2).mean()):.4f}")
    assert err.max() <= 2 * max(floor.max(), 2.5e-2)
    assert np.sqrt((err ** 2).mean()) <= 2 * max(np.sqrt((floor ** 2).mean()), 5e-3)
    # the greedy choice agrees wherever the oracle's top-2 margin exceeds the error
    for i in range(len(toks)):
        top = np.sort(want[i])[-2:]
        if top[1] - top[0] > 2 * err[i].max():
            assert int(np.argmax(gl[i])) == int(np.argmax(want[i]))
