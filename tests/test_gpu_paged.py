"""Paged target KV cache (kv_block > 0) on the GPU.

- Against the contiguous cache: a paged run differs only in where the target's keys and
  values live (blocks of kv_block slots handed out from a pool through a per-sequence block
  table), so prefill, every cycle and plain decoding must give bit-identical results:
  committed tokens, verify logits, trees, features, sampled draws.
- At the batch-64 Llama-3.1-8B EAGLE-3 configuration with 16-slot blocks (prompts of
  128..2048 tokens): greedy speculative output equals the GPU's own plain greedy decoding
  of every sequence exactly, and every accepted verify row's top-2 logit margin equals the
  plain step's bit for bit. The verify pass (1088 rows) and plain decoding (64 rows) sum
  each row in the same order: the GEMMs split k at the same points whatever the row count
  and the attention decomposes a row's keys by its position alone.
- At the same full-size model, paged and contiguous runs of eight of those sequences are
  bit-identical."""
import pytest
import torch

from eagle_speculative_decoding_cycle_gb300 import _lib as L
from eagle_speculative_decoding_cycle_gb300 import api, synth
from spec_plain import spec_vs_plain

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _record(wl, weights, prompts, kv_block, cycles, plain_steps, ref=None):
    B = len(prompts)
    D = wl.tree.depth
    max_ctx = max(len(p) for p in prompts) + (cycles + 2) * (D + 1) + plain_steps + 32
    eng = api.Engine(wl, weights, max_batch=B, max_ctx=max_ctx, kv_block=kv_block)
    eng.prefill([p.to(DEV) for p in prompts], ref)
    eng.set_debug(L.DEBUG_LOGITS)
    rec = {"state0": {k: v.clone() for k, v in eng.dump(L.DUMP_STATE).items()},
           "feat0": eng.dump(L.DUMP_FEATURES).clone(), "cycles": []}
    out = torch.zeros(B, D + 1, dtype=torch.int32, device=DEV)
    cnt = torch.zeros(B, dtype=torch.int32, device=DEV)
    for _ in range(cycles):
        eng.cycle(out, cnt)
        eng.sync()
        rec["cycles"].append((out.cpu().clone(), cnt.cpu().clone(), eng.dump(L.DUMP_VERIFY_LOGITS).clone(),
                              [t.clone() for t in eng.dump(L.DUMP_TREE)], eng.dump(L.DUMP_FEATURES).clone()))
    plain = torch.zeros(B, plain_steps, dtype=torch.int32, device=DEV)
    marg = torch.zeros(B, plain_steps, dtype=torch.float32, device=DEV)
    eng.decode_plain(plain_steps, plain, marg)
    eng.sync()
    rec["plain"] = plain.cpu()
    rec["state1"] = {k: v.clone() for k, v in eng.dump(L.DUMP_STATE).items()}
    if kv_block:
        _, tab_w, n_blocks, block = eng.kv_table()
        rec["table"] = (tab_w, n_blocks, block, eng.kv_view()[2])
    eng.close()
    return rec


def _same(a, b):
    assert torch.equal(a["feat0"], b["feat0"])
    for k in a["state0"]:
        assert torch.equal(a["state0"][k], b["state0"][k]), k
    assert len(a["cycles"]) == len(b["cycles"])
    for ca, cb in zip(a["cycles"], b["cycles"]):
        assert torch.equal(ca[0], cb[0]) and torch.equal(ca[1], cb[1])
        assert torch.equal(ca[2], cb[2])
        for ta, tb in zip(ca[3], cb[3]):
            assert torch.equal(ta, tb)
        assert torch.equal(ca[4], cb[4])
    assert torch.equal(a["plain"], b["plain"])
    for k in a["state1"]:
        assert torch.equal(a["state1"][k], b["state1"][k]), k


@pytest.mark.parametrize("name,kv_block,lens", [
    ("small-bf16-3L-H320", 16, (37, 20, 53)),       # ragged prompts: per-sequence prefill
    ("small-bf16-3L-H320", 8, (24, 24)),            # equal prompts: batched prefill
    ("small-bf16-eagle3-gqa", 16, (30, 9, 41)),     # GQA, EAGLE-3, sampling
    ("tiny-f32-2L-H256-V1024", 8, (33, 17)),        # fp32 model: the SIMT attention path
])
def test_paged_equals_contiguous(name, kv_block, lens):
    base = {w.name: w for w in (synth.SMALL_BF16, synth.SMALL_BF16_E3, synth.TINY)}[name]
    wl = base.replace(batch=len(lens), prompt_len=(min(lens), max(lens)))
    weights = {k: v.to(DEV) for k, v in synth.make_weights(wl, "cpu").items()}
    g = torch.Generator().manual_seed(1234)
    prompts = [torch.randint(0, wl.model.vocab, (n,), generator=g, dtype=torch.int64).to(torch.int32) for n in lens]
    a = _record(wl, weights, prompts, 0, cycles=4, plain_steps=5)
    b = _record(wl, weights, prompts, kv_block, cycles=4, plain_steps=5)
    _same(a, b)
    tab_w, n_blocks, block, cap = b["table"]
    assert block == kv_block and tab_w == -(-cap // kv_block) and n_blocks == len(lens) * tab_w


def test_paged_equals_contiguous_planted():
    """Planted mode (deep accepted paths, so compaction moves KV entries across block
    boundaries) with a reference taken from the contiguous engine's own plain decoding."""
    wl = synth.SMALL_BF16.replace(batch=3)
    weights = {k: v.to(DEV) for k, v in synth.make_weights(wl, "cpu").items()}
    g = torch.Generator().manual_seed(99)
    lens = (15, 31, 47)
    prompts = [torch.randint(0, wl.model.vocab, (n,), generator=g, dtype=torch.int64).to(torch.int32) for n in lens]
    eng = api.Engine(wl, weights, max_batch=3, max_ctx=max(lens) + 128)
    eng.prefill([p.to(DEV) for p in prompts])
    first = eng.dump(L.DUMP_STATE)["root_tok"].to(DEV)
    plain = torch.zeros(3, 60, dtype=torch.int32, device=DEV)
    eng.decode_plain(60, plain)
    eng.sync()
    eng.close()
    ref = torch.cat([first.view(3, 1).to(torch.int32), plain], 1).contiguous()
    a = _record(wl, weights, prompts, 0, cycles=6, plain_steps=3, ref=ref)
    b = _record(wl, weights, prompts, 16, cycles=6, plain_steps=3, ref=ref)
    _same(a, b)
    accepted = sum(int(c[1].sum()) for c in b["cycles"])
    assert accepted > 6 * 3 * 2, "planted mode should accept deep paths"


def test_batch64_llama31_8b_paged_lossless():
    """The batch-64 configuration at full size: greedy speculative decoding with the paged
    cache reproduces the GPU's plain greedy decoding of all 64 sequences bit for bit."""
    wl = synth.LLAMA31_8B_BS64
    weights = synth.make_weights(wl, device=DEV)
    prompts = synth.make_prompts(wl)
    rows, cycles = spec_vs_plain(wl, weights, prompts, 24, kv_block=16)
    print(f"batch 64: all {len(prompts)} sequences identical over 24 tokens; {rows} accepted verify rows "
          f"bit-identical to plain decoding over {cycles} cycles")


def test_8b_paged_equals_contiguous_full_size():
    """Eight of the batch-64 configuration's sequences at the full Llama-3.1-8B shape: the
    paged cache (16-slot blocks) and the contiguous cache give bit-identical runs."""
    wl = synth.LLAMA31_8B_BS64
    weights = synth.make_weights(wl, device=DEV)
    prompts = [p.cpu() for p in synth.make_prompts(wl)[:8]]
    sub = wl.replace(batch=8)
    a = _record(sub, weights, prompts, 0, cycles=3, plain_steps=3)
    b = _record(sub, weights, prompts, 16, cycles=3, plain_steps=3)
    _same(a, b)
