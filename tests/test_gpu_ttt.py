"""The EAGLE-3 training-time-test forward on the GPU against the oracle, row by row: for
each step s, the drafter outputs a^(s) of every source row (the self-fed features) and each
row's token cross-entropy, then the step's mean loss. Tolerances: the outputs are features,
held to the bound of the configuration (1e-4 fp32, 5e-2 bf16); a row's cross-entropy is the
difference of two logit-scale values (log-sum-exp minus the target's logit), each within
that bound, so it is held to twice it; the mean over rows to the bound itself."""
import numpy as np
import pytest
import torch

from eagle_speculative_decoding_cycle_gb300 import _lib as L
from eagle_speculative_decoding_cycle_gb300 import api, synth
from oracle.cycle import build_model
from oracle.ttt import cross_entropy, ttt_forward

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
def test_ttt_rows_and_losses_match_oracle(name, n, steps, tol):
    wl = {w.name: w for w in (synth.SMALL_BF16, synth.SMALL_BF16_E3, synth.TINY)}[name]
    weights = synth.make_weights(wl, "cpu")
    x = np.random.default_rng(17).integers(0, wl.model.vocab, n)
    M = build_model(synth.weights_to_numpy(weights), wl)
    want, outs = ttt_forward(M, x, steps)
    eng = api.Engine(wl, {k: v.to(DEV) for k, v in weights.items()})
    xd = torch.tensor(x, dtype=torch.int32, device=DEV)
    worst = []
    for s in range(1, steps + 1):
        # a run of s steps ends with step s, whose rows the debug view holds
        got = eng.ttt_forward(xd, s)
        eng.sync()
        a, ce = eng.dump(L.DUMP_TTT)
        a = a.double().numpy()
        ce = ce.double().numpy()
        wa = outs[s - 1]
        assert a.shape == wa.shape
        lg = M.logits(wa)
        wce = np.array([cross_entropy(lg[t], int(x[t + s + 1])) for t in range(wa.shape[0])])
        ea, ec = float(np.max(np.abs(a - wa))), float(np.max(np.abs(ce - wce)))
        el = abs(float(got[s - 1]) - want[s - 1])
        worst.append((s, round(ea, 6), round(ec, 6), round(el, 6)))
        assert ea < tol and ec < 2 * tol and el < tol
    print(name, "per step (max |a| error, max row CE error, mean loss error):", worst)
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
