"""The seeded input generators against the configuration table they stand for: model and
tree shapes, generated-node counts, weight bytes per verify pass and drafter step, prompt
lengths, and reproducibility of the seeded draws."""
import numpy as np
import pytest
import torch

from eagle_speculative_decoding_cycle_gb300 import synth

# (workload, hidden, layers, q heads, kv heads, head dim, ffn, vocab, k, D, m, N_gen)
TABLE = [
    (synth.TINY, 256, 2, 4, 4, 64, 688, 1024, 4, 4, 16, 52),
    (synth.LLAMA2_7B, 4096, 32, 32, 32, 128, 11008, 32000, 10, 6, 60, 510),
    (synth.LLAMA31_8B_SAMPLE, 4096, 32, 32, 8, 128, 14336, 128256, 10, 8, 60, 710),
    (synth.LLAMA_13B_LONG, 5120, 40, 40, 40, 128, 13824, 32000, 8, 6, 48, 328),
    (synth.LLAMA31_8B_BS64, 4096, 32, 32, 8, 128, 14336, 128256, 4, 5, 16, 68),
]


@pytest.mark.parametrize("row", TABLE, ids=lambda r: r[0].name)
def test_shapes_match_the_configuration_table(row):
    w, H, L, nq, nkv, d, F, V, k, D, m, n_gen = row
    s, t = w.model, w.tree
    assert (s.hidden, s.n_layers, s.n_heads, s.n_kv_heads, s.head_dim, s.ffn, s.vocab) == (H, L, nq, nkv, d, F, V)
    assert (t.topk, t.depth, t.m) == (k, D, m)
    assert t.n_gen == n_gen == k + (D - 1) * k * k


def _bytes(specs, prefix):
    return sum(int(np.prod(shape)) * 2 for name, shape, _ in specs if name.startswith(prefix))


@pytest.mark.parametrize("w,layers_gb,lm_gb,draft_layer_mb,fc_mb", [
    (synth.LLAMA2_7B, 12.95, 0.262, 405, 67),
    (synth.LLAMA31_8B_SAMPLE, 13.96, 1.05, 487, 101),
    (synth.LLAMA_13B_LONG, 25.38, 0.328, 634, 105),
])
def test_weight_bytes_match_the_table(w, layers_gb, lm_gb, draft_layer_mb, fc_mb):
    specs = synth.weight_specs(w.model, w.drafter)
    norms = [name for name, shape, std in specs if std == 0.0]
    assert all(len(shape) == 1 for name, shape, std in specs if name in norms)
    layers = _bytes([x for x in specs if x[2] != 0.0], "layers.")
    assert abs(layers / 1e9 - layers_gb) < 0.01
    lm = _bytes(specs, "lm_head")
    assert abs(lm / 1e9 - lm_gb) < 0.005
    draft = [x for x in specs if x[0].startswith("draft.") and x[2] != 0.0]
    assert abs(_bytes([x for x in draft if x[0] != "draft.fc"], "draft.") / 1e6 - draft_layer_mb) < 2
    assert abs(_bytes(draft, "draft.fc") / 1e6 - fc_mb) < 1


def test_batch64_prompts_are_seeded_uniform_lengths():
    w = synth.LLAMA31_8B_BS64
    a, b = synth.make_prompts(w), synth.make_prompts(w)
    assert len(a) == 64 == w.batch
    lens = [len(p) for p in a]
    assert all(128 <= n <= 2048 for n in lens)
    assert len(set(lens)) > 32                       # spread over the range, not one length
    assert all(torch.equal(x, y) for x, y in zip(a, b))
    assert all(int(p.min()) >= 0 and int(p.max()) < w.model.vocab for p in a)
    assert w.kv_block == 16


def test_fixed_length_prompts_and_weight_draws_are_reproducible():
    w = synth.SMALL_BF16
    (p,) = synth.make_prompts(w)
    assert len(p) == 40 and p.dtype == torch.int32
    w1, w2 = synth.make_weights(w), synth.make_weights(w)
    assert w1.keys() == w2.keys()
    assert all(torch.equal(w1[k], w2[k]) for k in w1)
    for name, shape, std in synth.weight_specs(w.model, w.drafter):
        t = w1[name]
        assert tuple(t.shape) == shape and t.dtype == torch.bfloat16
        if std == 0.0:
            assert bool((t == 1).all())
        else:
            assert abs(float(t.float().std()) / std - 1) < 0.1
    # another seed draws other weights
    other = synth.make_weights(w.replace(seed=w.seed + 1))
    assert not torch.equal(other["embed"], w1["embed"])
