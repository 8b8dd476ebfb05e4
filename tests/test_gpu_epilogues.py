"""The fused GEMM epilogues (RoPE + KV-cache write in the QKV projection, SwiGLU in the
gate/up projection) against the separate row kernels they replace: the same fp32
accumulator values go through the same arithmetic, so prefill, the drafter's candidates,
a cycle's tree, verify logits and committed tokens must be bit-identical."""
import os

import pytest
import torch

from eagle_speculative_decoding_cycle_gb300 import _lib as L
from eagle_speculative_decoding_cycle_gb300 import api, synth

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _run(wl, weights, prompts, max_batch=1, fuse: bool = True):
    saved = {k: os.environ.get(k) for k in ("EAGLE_FUSE_EPI",)}
    os.environ["EAGLE_FUSE_EPI"] = "3" if fuse else "0"
    try:
        eng = api.Engine(wl, weights, max_batch=max_batch)
    finally:
        for k, v in saved.items():
            if v is None:
                del os.environ[k]
            else:
                os.environ[k] = v
    eng.prefill([p.to(DEV) for p in prompts])
    eng.sync()
    st = eng.dump(L.DUMP_STATE)
    cand = eng.dump(L.DUMP_CAND)
    feat0 = eng.dump(L.DUMP_FEATURES).float().clone()
    eng.set_debug(L.DEBUG_LOGITS)
    B = len(prompts)
    out = torch.zeros(B, wl.tree.depth + 1, dtype=torch.int32, device=DEV)
    cnt = torch.zeros(B, dtype=torch.int32, device=DEV)
    eng.cycle(out, cnt)
    eng.sync()
    res = {"root": st["root_tok"].clone(), "cand_tok": cand[0].clone(), "cand_logc": cand[1].clone(),
           "tree": eng.dump(L.DUMP_TREE)[0].clone(), "logits": eng.dump(L.DUMP_VERIFY_LOGITS).clone(),
           "feat": eng.dump(L.DUMP_FEATURES).float().clone(), "feat0": feat0,
           "out": out.cpu(), "cnt": cnt.cpu()}
    eng.close()
    return res


WIDE = synth.SMALL_BF16.replace(
    name="wide-bf16-2L-H1024",
    model=synth.ModelShape(n_layers=2, hidden=1024, n_heads=8, n_kv_heads=8, head_dim=128, ffn=2816, vocab=1000,
                           rope_theta=1e4, dtype="bf16"))


@pytest.mark.parametrize("name", ["small-bf16-3L-H320", "small-bf16-eagle3-gqa", "wide-bf16-2L-H1024"])
def test_fused_epilogues_match_separate_kernels(name):
    """RoPE/KV-write and SwiGLU in the GEMM epilogues against the separate row kernels: the
    same fp32 values go through the same arithmetic, so every output is bit-identical."""
    wl = {w.name: w for w in (synth.SMALL_BF16, synth.SMALL_BF16_E3, WIDE)}[name]
    weights = {k: v.to(DEV) for k, v in synth.make_weights(wl, "cpu").items()}
    prompts = synth.make_prompts(wl)[:1]
    a = _run(wl, weights, prompts, fuse=True)
    b = _run(wl, weights, prompts, fuse=False)
    assert torch.equal(a["feat0"], b["feat0"])
    assert a["root"].tolist() == b["root"].tolist()
    assert torch.equal(a["cand_logc"], b["cand_logc"]) and torch.equal(a["cand_tok"], b["cand_tok"])
    assert torch.equal(a["tree"], b["tree"]) and torch.equal(a["logits"], b["logits"])
    assert a["out"].tolist() == b["out"].tolist() and a["cnt"].tolist() == b["cnt"].tolist()
