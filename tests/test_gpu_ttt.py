"""The EAGLE-3 training-time-test forward on the GPU against the oracle: per-step mean token
cross-entropy of the self-fed drafter pass with the TTT mask. Tolerances: 1e-4 for the fp32
model; 5e-2 for bf16 models (the loss is a difference of two logit-scale values, each within
the 5e-2 bf16 bound; the mean over rows only shrinks it)."""
import numpy as np
import pytest
import torch

from eagle_speculative_decoding_cycle_gb300 import _lib as L
from eagle_speculative_decoding_cycle_gb300 import api, synth
from oracle.cycle import build_model
from oracle.ttt import ttt_forward

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("name,n,steps,tol", [
    ("small-bf16-eagle3-gqa", 24, 3, 5e-2),
    ("small-bf16-3L-H320", 30, 4, 5e-2),
    ("tiny-f32-2L-H256-V1024", 20, 3, 1e-4),
])
def test_ttt_losses_match_oracle(name, n, steps, tol):
    wl = {w.name: w for w in (synth.SMALL_BF16, synth.SMALL_BF16_E3, synth.TINY)}[name]
    weights = synth.make_weights(wl, "cpu")
    x = np.random.default_rng(17).integers(0, wl.model.vocab, n)
    M = build_model(synth.weights_to_numpy(weights), wl)
    want, _ = ttt_forward(M, x, steps)
    eng = api.Engine(wl, {k: v.to(DEV) for k, v in weights.items()})
    got = eng.ttt_forward(torch.tensor(x, dtype=torch.int32, device=DEV), steps)
    eng.sync()
    got = got.cpu().double().numpy()
    print(name, "gpu", np.round(got, 5), "oracle", np.round(want, 5))
    assert np.max(np.abs(got - np.asarray(want))) < tol
    # the context works again after a prefill
    prompt = synth.make_prompts(wl)[0].to(DEV)
    eng.prefill([prompt])
    eng.cycle()
    eng.sync()
    eng.close()


def test_ttt_rejects_bad_arguments():
    wl = synth.SMALL_BF16_E3
    weights = {k: v.to(DEV) for k, v in synth.make_weights(wl, "cpu").items()}
    eng = api.Engine(wl, weights)
    x = torch.zeros(5, dtype=torch.int32, device=DEV)
    with pytest.raises(L.EagleError):
        eng.ttt_forward(x, 3)          # n < steps + 3
    with pytest.raises(L.EagleError):
        eng.ttt_forward(torch.zeros(4096, dtype=torch.int32, device=DEV), 2)   # longer than a prefill chunk
    eng.close()
