"""Failure detection without a GPU fault: each bounded device wait of the library, run on a
condition that nothing satisfies, gives up after its time limit, latches the timeout code
in the status word the host reads, and leaves the context usable for the next launch."""
import time

import numpy as np
import pytest
import torch

from eagle_speculative_decoding_cycle_gb300 import _lib as L
from eagle_speculative_decoding_cycle_gb300 import api

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
    assert np.max(np.abs(Y - ref)) <= 1e-3 * np.max(np.abs(ref)) + 1e-5


def test_wait_probe_rejects_bad_arguments():
    lib = L.lib()
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    assert lib.eagle_op_wait_probe(None, 2, None, err.data_ptr(), err.data_ptr()) == L.EAGLE_EINVAL
    assert lib.eagle_op_wait_probe(None, 1, None, err.data_ptr(), err.data_ptr()) == L.EAGLE_EINVAL
