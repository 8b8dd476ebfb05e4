"""The allocation-free GEMM entry point (eagle_op_gemm_noalloc) serves callers that cannot
allocate device memory where they run a projection, e.g. framework plugins handed only
their input and output buffers. Its scratch lives in the library's own device arrays.
This checks, through the C ABI, that two calls in a row agree with the allocating entry
point (eagle_op_gemm) within the GEMM tolerance of the other tests, and that requests
beyond its stated limit are refused. Kept in its own file so pytest collects it last."""
import numpy as np
import pytest
import torch

from eagle_speculative_decoding_cycle_gb300 import _lib as L
from eagle_speculative_decoding_cycle_gb300 import api

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _noalloc(W, X, epi, out):
    lib = L.lib()
    N, K = W.shape
    M = X.shape[0]
    return lib.eagle_op_gemm_noalloc(torch.cuda.current_stream().cuda_stream, W.data_ptr(), N, K, X.data_ptr(), M,
                                     epi, out.data_ptr(), out.stride(0))


@pytest.mark.parametrize("M,N,K", [(1, 4096, 4096), (10, 12288, 1024), (32, 5000, 328), (17, 640, 320)])
def test_noalloc_gemm_matches_allocating_gemm_twice(M, N, K):
    g = torch.Generator().manual_seed(M + N + K)
    X = torch.randn(M, K, generator=g).to(torch.bfloat16).to(DEV)
    W = (torch.randn(N, K, generator=g) * 0.05).to(torch.bfloat16).to(DEV)
    want = api.gemm(W, X, epi=0).cpu().double().numpy()
    mag = np.abs(X.cpu().double().numpy()) @ np.abs(W.cpu().double().numpy()).T
    for _ in range(2):          # two calls in a row share (and reuse) the library's scratch
        out = torch.full((M, N), float("nan"), dtype=torch.float32, device=DEV)
        assert _noalloc(W, X, 0, out) == L.EAGLE_OK
        torch.cuda.synchronize()
        got = out.cpu().double().numpy()
        assert np.all(np.abs(got - want) <= 1e-3 * mag + 1e-6)


def test_noalloc_gemm_refuses_beyond_limit():
    X = torch.zeros(33, 64, dtype=torch.bfloat16, device=DEV)
    W = torch.zeros(128, 64, dtype=torch.bfloat16, device=DEV)
    out = torch.zeros(33, 128, dtype=torch.float32, device=DEV)
    assert _noalloc(W, X, 0, out) == L.EAGLE_ECAPACITY
