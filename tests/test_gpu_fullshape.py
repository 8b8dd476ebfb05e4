"""Oracle parity at the full shapes of the 8B EAGLE-3 sampling, 13B long-context and batch-64
configurations, and bitwise losslessness at full size.

Lock step (the 8B EAGLE-3 model at temperature 1, the 13B EAGLE-1 model greedy), on a short
prompt (the first 32 tokens of the configuration's prompt, so that the fp64 oracle finishes in
minutes on the host):
- every cycle, the oracle's tree policy rerun on the GPU's own node table reproduces the
  GPU's expansions, kept set, flattened tree and ancestry mask bit for bit, and the
  acceptance walk on the GPU's own verify-head values reproduces its accepted path and bonus;
- in the first cycle the oracle, replaying the GPU's committed decisions (and verifying the
  GPU's tree where a near-tie in path values made its own differ), gives the verify logits of
  all m+1 rows. At full depth the GPU's logits must stay within twice the oracle's own
  fp32-accumulation floor on the same rows (the oracle with its matmuls summed in fp32 against
  itself in fp64; bf16 rounding points after every projection turn one-ulp fp32 differences
  into rounding flips that grow with depth), and within the bf16 bound 5e-2 in a 2-layer model
  of the same width.

Batch 64: four of the 64 sequences (the shortest prompts) after one paged cycle, the verify
logits of each sequence's deepest kept path against the oracle's plain causal forward of that
path, under the same full-depth floor.

Bitwise (GPU only): greedy speculative decoding at the full 7B shape (512-token prompt) and
the full 13B long-context shape (4096-token prompt) reproduces the GPU's own plain greedy
decoding token for token, with every accepted verify row's top-2 logit margin equal to the
plain step's."""
import dataclasses
import gc

import numpy as np
import pytest
import torch

from eagle_speculative_decoding_cycle_gb300 import _lib as L
from eagle_speculative_decoding_cycle_gb300 import api, synth
from oracle import model as om
from oracle import philox
from oracle.accept import greedy_walk, sample_walk
from oracle.cycle import OracleSeq, build_model
from oracle.model import KV
from spec_plain import check_tree_policy, spec_vs_plain

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
SHORT = 32


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _np(weights, n_layers=None):
    keep = (lambda k: not k.startswith("layers.") or int(k.split(".")[1]) < n_layers) if n_layers else (lambda k: True)
    return {k: v.to("cpu", torch.float32).numpy() for k, v in weights.items() if keep(k)}


def _layers(wl, n, fuse=None):
    d = wl.drafter if fuse is None else dataclasses.replace(wl.drafter, fuse_layers=fuse)
    return wl.replace(model=dataclasses.replace(wl.model, n_layers=n), drafter=d)


def _truncate(weights, n):
    return {k: v for k, v in weights.items() if not k.startswith("layers.") or int(k.split(".")[1]) < n}


def _fp32_floor(fn):
    """fn() with the oracle's matmuls summed in fp32 instead of fp64."""
    orig = om.mm
    om.mm = lambda a, w: (np.asarray(a, np.float32) @ np.asarray(w, np.float32).T).astype(np.float64)
    try:
        return fn()
    finally:
        om.mm = orig


def _walk(eng, wl, ft):
    """The acceptance walk on the GPU's own verify-head values (greedy argmax, or the
    point-mass rejection rule with the cycle's Philox draws)."""
    hid, hval, lse, spec = eng.dump(L.DUMP_VERIFY_HEAD)
    T = wl.tree.temperature
    if T == 0:
        return greedy_walk(ft, hid[:, 0].tolist())

    def p_child(row, tok):
        i = [int(ft.token[v]) for v in ft.children(row)].index(tok)
        return np.float32(np.exp(np.float32(spec[row, i]) * np.float32(1 / T) - np.float32(lse[row])))

    cyc = int(eng.dump(L.DUMP_STATE)["cycle"][0]) - 1
    return sample_walk(ft, p_child,
                       lambda row, i: philox.draw_uniform(wl.seed, philox.STREAM_ACCEPT, 0, cyc, i, row),
                       lambda row, ex: int(hid[row, 0]))


def lockstep(wl, weights, prompt, cycles, floor):
    """GPU cycles in lock step with the oracle; returns (max-abs logit error, floor max, error
    rms, floor rms, re-synced) of the first cycle."""
    D = wl.tree.depth
    eng = api.Engine(wl, weights, max_ctx=len(prompt) + (cycles + 2) * (D + 1) + 32)
    eng.prefill([prompt.to(DEV)])
    eng.set_debug(L.DEBUG_LOGITS)
    first = int(eng.dump(L.DUMP_STATE)["root_tok"][0])
    M = build_model(_np(weights), wl)
    o = OracleSeq(M, wl, capacity=len(prompt) + (cycles + 2) * (wl.tree.m + D + 2) + 32)
    o.prefill(prompt.numpy(), first=first)
    out = torch.zeros(1, D + 1, dtype=torch.int32, device=DEV)
    cnt = torch.zeros(1, dtype=torch.int32, device=DEV)
    res = None
    for c in range(cycles):
        n_before = int(eng.dump(L.DUMP_STATE)["ctx_len"][0])
        eng.cycle(out, cnt)
        eng.sync()
        t, ft, pos = check_tree_policy(eng, wl)
        assert pos.tolist() == (n_before + ft.depth).tolist()
        acc_len, bonus, path = eng.dump(L.DUMP_ACCEPT)
        gp, gb = _walk(eng, wl, ft)
        assert gp == path[0, :int(acc_len[0])].tolist() and gb == int(bonus[0])
        assert out[0, :int(cnt[0])].tolist() == [int(ft.token[r]) for r in gp] + [gb]
        if c == 0:
            o_f = o.fork() if floor else None
            plan = o.draft_and_verify()
            resync = not (plan.flat.token.tolist() == ft.token.tolist() and
                          plan.flat.parent.tolist() == ft.parent.tolist())
            if resync:
                plan = o.verify(t, ft)
            gl = eng.dump(L.DUMP_VERIFY_LOGITS).double().numpy()
            err = np.abs(gl - plan.logits)
            fl = np.abs(_fp32_floor(lambda: o_f.verify(t, ft)).logits - plan.logits) if floor else np.zeros(1)
            res = (float(err.max()), float(fl.max()), float(np.sqrt((err ** 2).mean())),
                   float(np.sqrt((fl ** 2).mean())), resync)
            o_f = None
    eng.close()
    return res


@pytest.mark.parametrize("base,fuse", [(synth.LLAMA31_8B_SAMPLE, (0, 1, 1)), (synth.LLAMA_13B_LONG, None)],
                         ids=["8b-eagle3-t1", "13b-eagle1"])
def test_full_width_two_layers_lockstep_within_bf16_tolerance(base, fuse):
    weights = synth.make_weights(_layers(base, 2, fuse), device=DEV)
    wl = _layers(base, 2, fuse).replace(prompt_len=(SHORT, SHORT))
    prompt = synth.make_prompts(base)[0][:SHORT]
    err, _, rms, _, resync = lockstep(wl, weights, prompt, cycles=2, floor=False)
    print(f"{base.name}, 2 layers: verify logits max {err:.4f} rms {rms:.5f} (re-synced: {resync})")
    assert err < 5e-2
    del weights
    gc.collect()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("base", [synth.LLAMA31_8B_SAMPLE, synth.LLAMA_13B_LONG], ids=["8b-eagle3-t1", "13b-eagle1"])
def test_full_depth_lockstep_within_fp32_floor(base):
    weights = synth.make_weights(base, device=DEV)
    wl = base.replace(prompt_len=(SHORT, SHORT))
    prompt = synth.make_prompts(base)[0][:SHORT]
    err, fl, rms, frms, resync = lockstep(wl, weights, prompt, cycles=2, floor=True)
    print(f"{base.name}, full depth: verify logits max {err:.4f} rms {rms:.5f}; fp32 floor max {fl:.4f} "
          f"rms {frms:.5f} (re-synced: {resync})")
    assert err <= 2 * max(fl, 2.5e-2)
    assert rms <= 2 * max(frms, 5e-3)
    del weights
    gc.collect()
    torch.cuda.empty_cache()


def test_batch64_four_sequences_against_the_oracle():
    wl = synth.LLAMA31_8B_BS64
    weights = synth.make_weights(wl, device=DEV)
    prompts = synth.make_prompts(wl)
    B, T1 = len(prompts), wl.tree.m + 1
    eng = api.Engine(wl, weights, max_batch=B, max_ctx=max(len(p) for p in prompts) + 64)
    eng.prefill([p.to(DEV) for p in prompts])
    eng.set_debug(L.DEBUG_LOGITS)
    eng.cycle()
    eng.sync()
    gl = eng.dump(L.DUMP_VERIFY_LOGITS).double().numpy()
    tok, pos, par, node, mask = eng.dump(L.DUMP_TREE)
    eng.close()
    M = build_model(_np(weights), wl.replace(drafter=synth.DrafterShape(kind=1)))
    s = wl.model
    picks = sorted(range(B), key=lambda b: len(prompts[b]))[:4]
    for b in picks:
        t_b, p_b = tok[b].tolist(), par[b].tolist()
        d = [0] * T1
        for r in range(1, T1):
            d[r] = d[p_b[r]] + 1
        chain = [int(np.argmax(d))]
        while p_b[chain[-1]] >= 0:
            chain.append(p_b[chain[-1]])
        chain = chain[::-1]
        seq = prompts[b].tolist() + [t_b[r] for r in chain]
        n = len(seq)

        def fwd():
            kv = KV.empty(s.n_layers, s.n_kv_heads, n, s.head_dim)
            p = np.arange(n)
            f, _ = M.target_rows(np.asarray(seq), p, kv, p, np.tril(np.ones((n, n), dtype=bool)))
            return M.logits(f[-len(chain):])

        want = fwd()
        floor = np.abs(_fp32_floor(fwd) - want)
        err = np.abs(gl[b * T1 + np.array(chain)] - want)
        print(f"batch 64, sequence {b} (prompt {len(prompts[b])}, path depth {len(chain) - 1}): max {err.max():.4f} "
              f"rms {np.sqrt((err ** 2).mean()):.5f}; fp32 floor max {floor.max():.4f} "
              f"rms {np.sqrt((floor ** 2).mean()):.5f}")
        assert err.max() <= 2 * max(floor.max(), 2.5e-2)
        assert np.sqrt((err ** 2).mean()) <= 2 * max(np.sqrt((floor ** 2).mean()), 5e-3)
    del weights
    gc.collect()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("wl,n_new", [(synth.LLAMA2_7B, 40), (synth.LLAMA_13B_LONG, 24)],
                         ids=["7b-prompt512", "13b-prompt4096"])
def test_full_size_greedy_spec_equals_plain_bitwise(wl, n_new):
    weights = synth.make_weights(wl, device=DEV)
    prompts = synth.make_prompts(wl)
    rows, cycles = spec_vs_plain(wl, weights, prompts, n_new)
    print(f"{wl.name}: {rows} accepted verify rows bit-identical to plain decoding over {cycles} cycles")
    assert rows > cycles
    del weights
    gc.collect()
    torch.cuda.empty_cache()
