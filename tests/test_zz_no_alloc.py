"""The allocation-free GEMM entry point (eagle_op_gemm_noalloc) serves callers that cannot
allocate device memory where they run a projection, e.g. framework plugins handed only
their input and output buffers. Its scratch lives in the library's own device arrays.
This checks, through the C ABI, that two calls in a row reproduce the allocating entry
point (eagle_op_gemm) bit for bit -- both run the same kernel with the same split-tile
schedule -- for each output mode (fp32 store, bf16 store, fp32 residual add), that the
shared status word reports no timeout afterwards, and that requests beyond its stated
limits are refused. Kept in its own file so pytest collects it last."""
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


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _noalloc(W, X, epi, out):
    lib = L.lib()
    N, K = W.shape
    M = X.shape[0]
    return lib.eagle_op_gemm_noalloc(_stream(), W.data_ptr(), N, K, X.data_ptr(), M, epi, out.data_ptr(),
                                     out.stride(0))


@pytest.mark.parametrize("epi", [0, 1, 2], ids=["f32", "bf16", "add"])
@pytest.mark.parametrize("M,N,K", [(1, 4096, 4096), (10, 12288, 1024), (32, 5000, 328), (17, 640, 320)])
def test_noalloc_gemm_matches_allocating_gemm_twice(M, N, K, epi):
    g = torch.Generator().manual_seed(M + N + K + epi)
    X = torch.randn(M, K, generator=g).to(torch.bfloat16).to(DEV)
    W = (torch.randn(N, K, generator=g) * 0.05).to(torch.bfloat16).to(DEV)
    odt = torch.bfloat16 if epi == 1 else torch.float32
    base = torch.randn(M, N, generator=g).to(DEV)
    want = base.clone() if epi == 2 else torch.zeros(M, N, dtype=odt, device=DEV)
    api.gemm(W, X, epi=epi, out=want)
    for _ in range(2):          # two calls in a row share (and reuse) the library's scratch
        out = base.clone() if epi == 2 else torch.full((M, N), float("nan"), dtype=odt, device=DEV)
        assert _noalloc(W, X, epi, out) == L.EAGLE_OK
        torch.cuda.synchronize()
        assert torch.equal(out, want)
    assert L.lib().eagle_op_gemm_noalloc_status(_stream()) == L.EAGLE_OK


def test_noalloc_gemm_refuses_beyond_limits():
    lib = L.lib()
    X = torch.zeros(33, 64, dtype=torch.bfloat16, device=DEV)
    W = torch.zeros(128, 64, dtype=torch.bfloat16, device=DEV)
    out = torch.zeros(33, 128, dtype=torch.float32, device=DEV)
    assert _noalloc(W, X, 0, out) == L.EAGLE_ECAPACITY          # more than 32 rows
    # more than 8192 output tiles (128 features each): refused on the host, nothing launched
    N = 8192 * 128 + 1
    Wb = torch.zeros(N, 8, dtype=torch.bfloat16, device=DEV)
    Xs = torch.zeros(1, 8, dtype=torch.bfloat16, device=DEV)
    ob = torch.zeros(1, N, dtype=torch.float32, device=DEV)
    assert lib.eagle_op_gemm_noalloc(_stream(), Wb.data_ptr(), N, 8, Xs.data_ptr(), 1, 0, ob.data_ptr(),
                                     N) == L.EAGLE_ECAPACITY
    assert lib.eagle_op_gemm_noalloc(_stream(), Wb.data_ptr(), N, 8, Xs.data_ptr(), 1, 3, ob.data_ptr(),
                                     N) == L.EAGLE_EINVAL   # the fused LM head is not an output mode here
