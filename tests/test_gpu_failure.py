"""Failure detection without a GPU fault.

- Each bounded device wait of the library, run on a condition that nothing satisfies,
  gives up after its time limit, latches the timeout code in the status word the host
  reads, and leaves the context usable for the next launch.
- A token id outside the vocabulary in a prompt is caught by the kernels' own bounds
  checks (the row is skipped, never read out of range) and reported as EAGLE_EDEVICE by
  the next status read; the context then runs a correct cycle.
- The host fault hooks (EAGLE_FAULT=prefill|cycle) fail the named call on the host,
  before any launch, and the context keeps working once they are lifted."""
import os
import time

import numpy as np
import pytest
import torch

from eagle_speculative_decoding_cycle_gb300 import _lib as L
from eagle_speculative_decoding_cycle_gb300 import api, synth

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
DEVERR_TIMEOUT = 1


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("kind", [0, 1], ids=["mbarrier", "grid-counter"])
def test_bounded_wait_times_out_and_reports(kind):
    lib = L.lib()
    counter = torch.zeros(1, dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    result = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    rc = lib.eagle_op_wait_probe(torch.cuda.current_stream().cuda_stream, kind, counter.data_ptr(),
                                 err.data_ptr(), result.data_ptr())
    assert rc == L.EAGLE_OK
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert int(result[0]) == 0, "the wait must give up"
    assert int(err[0]) == DEVERR_TIMEOUT
    assert 1.5 < waited < 30.0, waited          # the library's limit is 2 s
    # the context is still usable: a tensor-core GEMM right after gives the right answer
    g = torch.Generator().manual_seed(1)
    X = torch.randn(17, 256, generator=g).to(torch.bfloat16)
    W = (torch.randn(384, 256, generator=g) * 0.05).to(torch.bfloat16)
    Y = api.gemm(W.to(DEV), X.to(DEV)).cpu().double().numpy()
    ref = X.double().numpy() @ W.double().numpy().T
    mag = np.abs(X.double().numpy()) @ np.abs(W.double().numpy()).T
    assert np.all(np.abs(Y - ref) <= 1e-5 * mag + 1e-6)


def test_wait_probe_rejects_bad_arguments():
    lib = L.lib()
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    assert lib.eagle_op_wait_probe(None, 2, None, err.data_ptr(), err.data_ptr()) == L.EAGLE_EINVAL
    assert lib.eagle_op_wait_probe(None, 1, None, err.data_ptr(), err.data_ptr()) == L.EAGLE_EINVAL


def _engine(wl):
    weights = {k: v.to(DEV) for k, v in synth.make_weights(wl, "cpu").items()}
    return api.Engine(wl, weights), synth.make_prompts(wl)[0].to(DEV)


def _cycle_tokens(eng, wl, n=3):
    D = wl.tree.depth
    out = torch.zeros(1, D + 1, dtype=torch.int32, device=DEV)
    cnt = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = []
    for _ in range(n):
        eng.cycle(out, cnt)
        eng.sync()
        got += out[0, :int(cnt[0])].tolist()
    return got


@pytest.mark.parametrize("wl", [synth.SMALL_BF16, synth.SMALL_BF16_E3], ids=["eagle1", "eagle3"])
def test_out_of_range_prompt_token_reports_edevice(wl):
    eng, prompt = _engine(wl)
    eng.prefill([prompt])
    ref = _cycle_tokens(eng, wl)
    bad = prompt.clone()
    bad[len(bad) // 2] = wl.model.vocab          # one past the last id
    eng.prefill([bad])
    with pytest.raises(L.EagleError) as e:
        eng.sync()
    assert e.value.code == L.EAGLE_EDEVICE
    eng.sync()                                   # the status word was cleared by the read
    eng.prefill([prompt])
    assert _cycle_tokens(eng, wl) == ref
    eng.close()


@pytest.mark.parametrize("hook", ["prefill", "cycle"])
def test_host_fault_hooks_fail_the_call_and_leave_the_context_usable(hook, monkeypatch):
    wl = synth.SMALL_BF16
    eng, prompt = _engine(wl)
    eng.prefill([prompt])
    ref = _cycle_tokens(eng, wl)
    eng.prefill([prompt])
    monkeypatch.setenv("EAGLE_FAULT", hook)
    with pytest.raises(L.EagleError) as e:
        if hook == "prefill":
            eng.prefill([prompt])
        else:
            eng.cycle()
    assert e.value.code == L.EAGLE_ECUDA
    monkeypatch.delenv("EAGLE_FAULT")
    eng.sync()
    if hook == "prefill":
        eng.prefill([prompt])
    assert _cycle_tokens(eng, wl) == ref
    eng.close()
