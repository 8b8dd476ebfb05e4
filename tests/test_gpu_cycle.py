"""End-to-end GPU parity of prefill, the draft-and-verify cycle and plain decoding.

- Index work is checked in lock step: after every GPU cycle the oracle's tree policy
  is rerun on the GPU's own path values and its acceptance walk on the GPU's own verify
  head outputs; expansion order, kept set, flattened tree, mask, accepted path and
  bonus must agree bit for bit.
- Floats: verify-row features/logits against the oracle, 1e-4 (fp32 model) or 5e-2
  (bf16 model) max-abs.
- Greedy losslessness: speculative output equals plain greedy decoding (the GPU's own
  decode_plain and the oracle's)."""
import dataclasses

import numpy as np
import pytest
import torch

from eagle_speculative_decoding_cycle_gb300 import _lib as L
from eagle_speculative_decoding_cycle_gb300 import api, synth
from oracle import philox
from oracle.accept import greedy_walk, sample_walk
from oracle.cycle import OracleSeq, build_model, plain_decode
from oracle.tree import NodeTable, flatten, rerank, select_expand, static_plan
from spec_plain import check_tree_policy, gpu_table, spec_vs_plain

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def setup(wl, planted=True, extra=8):
    weights = synth.make_weights(wl, "cpu")
    M = build_model(synth.weights_to_numpy(weights), wl)
    prompt = synth.make_prompts(wl)[0]
    R = plain_decode(M, wl, prompt.numpy(), wl.new_tokens + wl.tree.depth + extra) if planted else None
    eng = api.Engine(wl, {k: v.to(DEV) for k, v in weights.items()})
    return weights, M, prompt, R, eng


def run_lockstep(wl, n_cycles=None, planted=True, check_feats_tol=None):
    weights, M, prompt, R, eng = setup(wl, planted)
    ref = None if R is None else torch.tensor([R], dtype=torch.int32, device=DEV)
    eng.prefill([prompt.to(DEV)], ref)
    eng.set_debug(L.DEBUG_LOGITS)
    o = OracleSeq(M, wl)
    o.prefill(prompt.numpy(), R)
    st = eng.dump(L.DUMP_STATE)
    assert int(st["root_tok"][0]) == o.committed[0]
    D = wl.tree.depth
    out = torch.zeros(1, D + 1, dtype=torch.int32, device=DEV)
    cnt = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = [int(st["root_tok"][0])]
    stats = {"cycles": 0, "tree_match": 0, "max_feat_err": 0.0, "max_logit_err": 0.0, "accepted": []}
    T = wl.tree.temperature
    while len(got) < wl.new_tokens and (n_cycles is None or stats["cycles"] < n_cycles):
        n_before = int(eng.dump(L.DUMP_STATE)["ctx_len"][0])
        eng.cycle(out, cnt)
        eng.sync()
        t, ft, pos = check_tree_policy(eng, wl)
        assert pos.tolist() == (n_before + ft.depth).tolist()
        acc_len, bonus, path = eng.dump(L.DUMP_ACCEPT)
        L_ = int(acc_len[0])
        hid, hval, lse, spec = eng.dump(L.DUMP_VERIFY_HEAD)
        if T == 0:
            gp, gb = greedy_walk(ft, hid[:, 0].tolist())
        else:
            def p_child(row, tok):
                i = [int(ft.token[v]) for v in ft.children(row)].index(tok)
                return np.float32(np.exp(np.float32(spec[row, i]) * np.float32(1 / T) - np.float32(lse[row])))

            cyc = int(eng.dump(L.DUMP_STATE)["cycle"][0]) - 1
            gp, gb = sample_walk(ft, p_child,
                                 lambda row, i: philox.draw_uniform(wl.seed, philox.STREAM_ACCEPT, 0, cyc, i, row),
                                 lambda row, ex: int(hid[row, 0]))
        assert gp == path[0, :L_].tolist() and gb == int(bonus[0])
        new = out[0, :int(cnt[0])].tolist()
        assert new == [int(ft.token[r]) for r in gp] + [gb]
        # oracle in lock step: it drafts its own tree; the same tree -> compare the verify
        # rows' floats. A different tree (a near-tie in path values decided the other way in
        # fp32 and fp64) is counted, and the oracle then verifies the GPU's tree instead, so
        # the floats are still compared; either way the oracle commits the GPU's decisions
        plan = o.draft_and_verify()
        if plan.flat.token.tolist() == ft.token.tolist() and plan.flat.parent.tolist() == ft.parent.tolist():
            stats["tree_match"] += 1
        else:
            stats["resync"] = stats.get("resync", 0) + 1
            plan = o.verify(t, ft)
        gl = eng.dump(L.DUMP_VERIFY_LOGITS).double().numpy()
        stats["max_logit_err"] = max(stats["max_logit_err"], float(np.max(np.abs(gl - plan.logits))))
        gf = eng.dump(L.DUMP_FEATURES).double().numpy()
        stats["max_feat_err"] = max(stats["max_feat_err"], float(np.max(np.abs(gf - plan.feats))))
        o.commit(plan, gp, gb)
        got += new
        stats["cycles"] += 1
        stats["accepted"].append(L_)
    eng.close()
    return got, R, stats


def test_tiny_fp32_lockstep_and_lossless():
    wl = synth.TINY
    got, R, st = run_lockstep(wl)
    N = wl.new_tokens
    assert got[:N] == R[:N]                     # greedy speculative == plain greedy
    assert st["tree_match"] == st["cycles"]     # same trees every cycle
    assert st["max_logit_err"] < 1e-4 and st["max_feat_err"] < 1e-4
    assert max(st["accepted"]) >= 2


# static (EAGLE-1) trees on the tiny model (k = 4, D = 4): a chain, and a 16-node shape
TINY_CHAIN = synth.TINY.replace(tree=synth.TreeShape(topk=4, depth=4, m=4, planted_p=0.8,
                                                     static_parent=(-1, 0, 1, 2), static_rank=(0, 0, 0, 0)))
TINY_STATIC = synth.TINY.replace(tree=synth.TreeShape(
    topk=4, depth=4, m=16, planted_p=0.8,
    static_parent=(-1, -1, -1, 0, 0, 0, 1, 1, 2, 3, 3, 4, 6, 9, 9, 10),
    static_rank=(0, 1, 2, 0, 1, 2, 0, 1, 0, 0, 1, 0, 0, 0, 1, 0)))


@pytest.mark.parametrize("wl", [TINY_CHAIN, TINY_STATIC], ids=["chain", "static16"])
def test_tiny_fp32_static_tree_lockstep_and_lossless(wl):
    """The static policy: every cycle the GPU expands the planned rows and verifies exactly
    the topology (checked against the oracle's plan on the GPU's own node table), the
    floats match the oracle in lock step, and greedy output stays lossless."""
    got, R, st = run_lockstep(wl)
    N = wl.new_tokens
    assert got[:N] == R[:N]
    assert st["tree_match"] == st["cycles"]
    assert st["max_logit_err"] < 1e-4 and st["max_feat_err"] < 1e-4
    assert max(st["accepted"]) >= 2


def test_static_tree_can_be_switched_off():
    """set_static_tree with an empty topology restores the dynamic policy: the run then
    equals a context created without a static tree."""
    wl = TINY_STATIC
    weights, M, prompt, R, eng = setup(wl)
    dyn = synth.TINY.replace(tree=synth.TreeShape(topk=4, depth=4, m=16, planted_p=0.8))
    eng2 = api.Engine(dyn, {k: v.to(DEV) for k, v in weights.items()})
    eng.set_static_tree([], [])
    ref = torch.tensor([R], dtype=torch.int32, device=DEV)
    outs = []
    for e in (eng, eng2):
        e.prefill([prompt.to(DEV)], ref)
        out = torch.zeros(1, 5, dtype=torch.int32, device=DEV)
        cnt = torch.zeros(1, dtype=torch.int32, device=DEV)
        seq = []
        for _ in range(4):
            e.cycle(out, cnt)
            e.sync()
            seq.append((out.cpu().clone(), cnt.cpu().clone(), [x.clone() for x in e.dump(L.DUMP_TREE)]))
        outs.append(seq)
        e.close()
    for (oa, ca, ta), (ob, cb, tb) in zip(*outs):
        assert torch.equal(oa, ob) and torch.equal(ca, cb)
        assert all(torch.equal(x, y) for x, y in zip(ta, tb))


def test_tiny_fp32_plain_decode_matches_oracle():
    wl = synth.TINY
    weights, M, prompt, R, eng = setup(wl)
    eng.prefill([prompt.to(DEV)])
    n = 40
    out = torch.zeros(1, n, dtype=torch.int32, device=DEV)
    first = int(eng.dump(L.DUMP_STATE)["root_tok"][0])
    eng.decode_plain(n, out)
    eng.sync()
    assert [first] + out[0].tolist() == R[:n + 1]
    eng.close()


def test_small_bf16_lockstep_and_lossless():
    wl = synth.SMALL_BF16
    got, R, st = run_lockstep(wl)
    N = wl.new_tokens
    # Greedy choices are exact up to the first position whose fp64 top-2 margin is inside
    # bf16 rounding noise: there either token is the argmax of a correctly rounded bf16
    # forward, and the continuations may part.
    k = first_near_tie(wl, N)
    assert k >= 10
    assert got[:k] == R[:k]
    assert st["tree_match"] >= 1
    assert st["tree_match"] + st.get("resync", 0) == st["cycles"]     # floats compared every cycle
    assert st["max_logit_err"] < 5e-2 and st["max_feat_err"] < 5e-2
    print(f"bf16 lock step: {st['cycles']} cycles, {st.get('resync', 0)} re-synced on the GPU's tree, "
          f"max logit error {st['max_logit_err']:.4f}, max feature error {st['max_feat_err']:.4f}")


NEAR_TIE = 1e-2


def first_near_tie(wl, n):
    """First greedy position whose oracle (fp64) top-2 logit margin is below NEAR_TIE."""
    M = build_model(synth.weights_to_numpy(synth.make_weights(wl, "cpu")), wl)
    margins = []
    plain_decode(M, wl, synth.make_prompts(wl)[0].numpy(), n, margins=margins)
    small = [i for i, m in enumerate(margins[:n]) if m < NEAR_TIE]
    return small[0] if small else n


def _first_diff(a, b):
    n = min(len(a), len(b))
    return next((i for i in range(n) if a[i] != b[i]), n)


@pytest.mark.parametrize("wl,kv_block,lens", [
    (synth.SMALL_BF16.replace(new_tokens=48), 0, (40,)),
    (synth.SMALL_BF16_E3.replace(tree=synth.TreeShape(topk=4, depth=5, m=14, planted_p=0.8), new_tokens=40), 0, (24,)),
    # a longer context: several key splits in every verify and plain row
    (synth.SMALL_BF16.replace(new_tokens=40), 0, (700,)),
    # batched, ragged, paged
    (synth.SMALL_BF16_E3.replace(tree=synth.TreeShape(topk=4, depth=5, m=14, planted_p=0.8), new_tokens=30), 16,
     (37, 130, 9)),
], ids=["eagle1", "eagle3-gqa", "eagle1-ctx700", "eagle3-batch3-paged"])
def test_bf16_spec_equals_gpu_plain_bitwise(wl, kv_block, lens):
    """Greedy speculative output equals the GPU's own plain greedy decoding exactly, and every
    accepted verify row's logits (through their top-2 margin) equal the plain step's: the
    verify pass and plain decoding sum every row in the same order."""
    weights = {k: v.to(DEV) for k, v in synth.make_weights(wl, "cpu").items()}
    g = torch.Generator().manual_seed(sum(lens))
    prompts = [torch.randint(0, wl.model.vocab, (n,), generator=g, dtype=torch.int64).to(torch.int32) for n in lens]
    rows, cycles = spec_vs_plain(wl, weights, prompts, wl.new_tokens, kv_block=kv_block)
    print(f"{wl.name}: {rows} accepted rows bit-identical over {cycles} cycles")
    assert rows > cycles * len(lens)        # planted mode accepts paths deeper than the root


def test_bf16_plain_decode_matches_oracle_up_to_near_ties():
    wl = synth.SMALL_BF16
    weights = synth.make_weights(wl, "cpu")
    M = build_model(synth.weights_to_numpy(weights), wl)
    prompt = synth.make_prompts(wl)[0]
    margins = []
    R = plain_decode(M, wl, prompt.numpy(), 40, margins=margins)
    eng = api.Engine(wl, {k: v.to(DEV) for k, v in weights.items()})
    eng.prefill([prompt.to(DEV)])
    out = torch.zeros(1, 39, dtype=torch.int32, device=DEV)
    first = int(eng.dump(L.DUMP_STATE)["root_tok"][0])
    eng.decode_plain(39, out)
    eng.sync()
    got = [first] + out[0].tolist()
    i = _first_diff(got, R)
    assert i == len(R) or margins[i] < NEAR_TIE, (i, margins[i])
    eng.close()


def test_eagle3_sampling_lockstep():
    wl = synth.SMALL_BF16_E3
    got, R, st = run_lockstep(wl, planted=False)
    assert st["cycles"] >= 3
    assert st["max_logit_err"] < 5e-2 and st["max_feat_err"] < 5e-2


def test_eagle3_greedy_lossless():
    wl = synth.SMALL_BF16_E3.replace(tree=synth.TreeShape(topk=4, depth=5, m=14, temperature=0.0, planted_p=0.8))
    got, R, st = run_lockstep(wl)
    N = wl.new_tokens
    assert got[:N] == R[:N]
    assert max(st["accepted"]) >= 2


def test_graph_replay_equals_eager():
    wl = synth.TINY
    weights, M, prompt, R, eng = setup(wl)
    ref = torch.tensor([R], dtype=torch.int32, device=DEV)
    D = wl.tree.depth
    res = []
    for graph in (False, True):
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            e2 = api.Engine(wl, {k: v.to(DEV) for k, v in weights.items()}, stream=s)
            e2.set_graph(graph)
            e2.prefill([prompt.to(DEV)], ref)
            out = torch.zeros(1, D + 1, dtype=torch.int32, device=DEV)
            cnt = torch.zeros(1, dtype=torch.int32, device=DEV)
            toks = []
            for _ in range(10):
                e2.cycle(out, cnt)
                e2.sync()
                toks += out[0, :int(cnt[0])].tolist()
            res.append(toks)
            e2.close()
    assert res[0] == res[1]
    eng.close()


def test_capacity_error_before_launch():
    wl = synth.TINY
    weights, M, prompt, R, _ = setup(wl, planted=False)
    eng = api.Engine(wl, {k: v.to(DEV) for k, v in weights.items()}, max_ctx=40)
    eng.prefill([prompt.to(DEV)])
    with pytest.raises(L.EagleError) as e:
        for _ in range(10):
            eng.cycle()
    assert e.value.code == L.EAGLE_ECAPACITY
    eng.sync()
    eng.close()


def test_finished_sequences_are_masked_out_of_later_cycles():
    """Per-sequence generation limits in a batch: each sequence emits exactly its limit (the
    last cycle's surplus dropped), its tokens equal its plain greedy continuation, and once
    finished it commits nothing and its state stays as it was while the others go on."""
    wl = synth.SMALL_BF16_E3.replace(tree=synth.TreeShape(topk=4, depth=5, m=14, planted_p=0.8), batch=3)
    weights = {k: v.to(DEV) for k, v in synth.make_weights(wl, "cpu").items()}
    g = torch.Generator().manual_seed(7)
    prompts = [torch.randint(0, wl.model.vocab, (n,), generator=g, dtype=torch.int64).to(torch.int32).to(DEV)
               for n in (20, 33, 41)]
    limits = [6, 40, 15]
    D = wl.tree.depth
    eng = api.Engine(wl, weights, max_batch=3, max_ctx=41 + 160)
    eng.prefill(prompts)
    first = eng.dump(L.DUMP_STATE)["root_tok"][:3].to(torch.int32)
    plain = torch.zeros(3, 60, dtype=torch.int32, device=DEV)
    eng.decode_plain(60, plain)
    eng.sync()
    ref = torch.cat([first.view(3, 1).to(DEV), plain], 1).contiguous()
    eng.prefill(prompts, ref)
    eng.set_stop(limits)
    got = [[int(first[b])] for b in range(3)]
    out = torch.zeros(3, D + 1, dtype=torch.int32, device=DEV)
    cnt = torch.zeros(3, dtype=torch.int32, device=DEV)
    frozen = {}
    stats = eng.new_stats()
    for _ in range(40):
        before = {k: v.clone() for k, v in eng.dump(L.DUMP_STATE).items()}
        eng.cycle(out, cnt, stats)
        eng.sync()
        after = eng.dump(L.DUMP_STATE)
        o, c = out.cpu(), cnt.cpu()
        # the cycle's statistics: the batch's counters and the device clock per phase
        st, acc = api.read_stats(stats), eng.dump(L.DUMP_ACCEPT)[0].cpu()
        live = [b for b in range(3) if int(c[b]) > 0]
        assert (st["batch"], st["active"], st["committed"], st["verify_rows"]) == (3, len(live), int(c.sum()), 15)
        assert st["accepted"] == sum(int(acc[b]) for b in live)
        assert st["max_accepted"] == max([int(acc[b]) for b in live] + [0])
        assert all(t > 0 for t in st["phase_us"].values()), st
        assert abs(sum(st["phase_us"].values()) - st["cycle_us"]) < 1e-3
        for b in range(3):
            if len(got[b]) >= limits[b]:
                assert int(c[b]) == 0
                for key in ("ctx_len", "committed", "root_tok"):
                    assert int(after[key][b]) == int(before[key][b]), (b, key)
                frozen[b] = True
            got[b] += o[b, :int(c[b])].tolist()
        if all(len(got[b]) >= limits[b] for b in range(3)) and len(frozen) == 3:
            break
    for b in range(3):
        assert len(got[b]) == limits[b], (b, len(got[b]))
        assert got[b] == ref[b, :limits[b]].tolist()
    assert len(frozen) == 3
    eng.set_stop([])
    eng.cycle(out, cnt)
    eng.sync()
    assert all(int(x) >= 1 for x in cnt.cpu())          # limits removed: every sequence moves again
    eng.close()


@pytest.mark.parametrize("temperature", [0.0, 1.0], ids=["greedy", "sampling"])
def test_tree_budget_change_between_cycles(temperature):
    """Lowering k and m between cycles gives exactly the cycles of a context created with the
    lower values: the root candidates are kept at the created k in rank order and the tree
    takes the first k of them. Raising either beyond the created values is refused."""
    big = synth.SMALL_BF16.replace(tree=synth.TreeShape(topk=5, depth=4, m=12, temperature=temperature,
                                                        planted_p=0.8))
    small = big.replace(tree=dataclasses.replace(big.tree, topk=3, m=8))
    weights = {k: v.to(DEV) for k, v in synth.make_weights(big, "cpu").items()}
    prompt = synth.make_prompts(big)[0].to(DEV)
    runs = []
    for wl, switch in ((big, True), (small, False)):
        eng = api.Engine(wl, weights)
        eng.prefill([prompt])
        if switch:
            with pytest.raises(L.EagleError):
                eng.set_tree_budget(6, 8)
            with pytest.raises(L.EagleError):
                eng.set_tree_budget(3, 13)
            eng.set_tree_budget(3, 8)
        out = torch.zeros(1, wl.tree.depth + 1, dtype=torch.int32, device=DEV)
        cnt = torch.zeros(1, dtype=torch.int32, device=DEV)
        rec = []
        for _ in range(6):
            eng.cycle(out, cnt)
            eng.sync()
            rec.append((out[0, :int(cnt[0])].tolist(), [t.clone() for t in eng.dump(L.DUMP_TREE)]))
        runs.append(rec)
        eng.close()
    for (ta, tra), (tb, trb) in zip(*runs):
        assert ta == tb
        assert all(torch.equal(x, y) for x, y in zip(tra, trb))


def test_phase_timing_and_graph_stats():
    """Per-phase timing: CUDA events at the phase boundaries of profiled eager cycles (each
    phase takes time; the verify phase is what eagle_profile_verify reports), and the
    device-clock statistics of graph-replayed cycles (counters equal the outputs)."""
    wl = synth.SMALL_BF16_E3.replace(tree=synth.TreeShape(topk=4, depth=5, m=14, planted_p=0.8), batch=2)
    weights = {k: v.to(DEV) for k, v in synth.make_weights(wl, "cpu").items()}
    g = torch.Generator().manual_seed(3)
    prompts = [torch.randint(0, wl.model.vocab, (n,), generator=g, dtype=torch.int64).to(torch.int32).to(DEV)
               for n in (24, 24)]
    D = wl.tree.depth
    stream = torch.cuda.Stream()
    eng = api.Engine(wl, weights, max_batch=2, max_ctx=24 + 12 * (D + 1) + 16, stream=stream)
    with torch.cuda.stream(stream):
        eng.prefill(prompts)
        eng.profile_begin(0)
        for _ in range(3):
            eng.cycle()
        eng.profile_end()
    n, phases = eng.profile_phases()
    nv, vms = eng.profile_verify()
    assert n == nv == 3
    assert list(phases) == list(L.PHASES) and all(ms > 0 for ms in phases.values()), phases
    assert phases["verify"] == vms
    out = torch.zeros(2, D + 1, dtype=torch.int32, device=DEV)
    cnt = torch.zeros(2, dtype=torch.int32, device=DEV)
    stats = eng.new_stats()
    with torch.cuda.stream(stream):
        eng.set_graph(True)
        for _ in range(3):
            eng.cycle(out, cnt, stats)
            eng.sync()
            st, acc = api.read_stats(stats), eng.dump(L.DUMP_ACCEPT)[0].cpu()
            c = cnt.cpu()
            assert (st["batch"], st["active"], st["committed"]) == (2, 2, int(c.sum()))
            assert st["accepted"] == int(acc[:2].sum()) == int(c.sum()) - 2
            assert all(t > 0 for t in st["phase_us"].values()), st
        eng.set_graph(False)
    eng.close()
