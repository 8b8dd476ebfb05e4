// Allocation-free entry point of the tensor-core projection GEMM.
//
// The regular entry point (eagle_op_gemm) takes its split-tile scratch from the caller,
// who must allocate it. Some callers cannot allocate device memory at the point where
// they run a GEMM: code inside a host framework whose execution phase forbids
// allocation (plugins that only receive input and output buffers), code driven from a
// context where cudaMalloc would synchronise or is not permitted, or runtimes that pool
// all device memory up front. For them this variant keeps its scratch in file-scope
// __device__ arrays that exist on every GPU the library is loaded on, for as long as
// the process lives, so a call needs only its inputs and outputs.
#include <mutex>

#include "../../include/eagle.h"
#include "../../include/eagle_ops.h"
#include "common.cuh"
#include "kernels.h"

// Limits of this variant: at most 32 rows (tokens), hence at most 32 accumulator
// columns per tile; at most 192 CTAs (one per SM) and 8192 output tiles.
constexpr int kNoallocMaxRows = 32;
constexpr int kNoallocMaxCtas = 192;
constexpr int kNoallocMaxTiles = 8192;

// Split-tile partial sums, [cta][2 slots][32 columns][128 rows] fp32 (6 MiB), and the
// per-tile counters through which a split tile's later contributors hand their partial
// sums to the CTA that finishes it (32 KiB).
static __device__ __align__(256) float g_noalloc_partials[kNoallocMaxCtas * 2 * kNoallocMaxRows * 128];
static __device__ __align__(256) int g_noalloc_tickets[kNoallocMaxTiles];
// Status word: a bounded device wait that gives up (a split tile whose partial sums never
// arrive) records the timeout here instead of returning silently. It is sticky across
// calls until eagle_op_gemm_noalloc_status reads and clears it.
static __device__ __align__(256) int g_noalloc_status[4];

namespace {

struct DeviceScratch {
  float* partials = nullptr;
  int* tickets = nullptr;
  int* status = nullptr;
  bool ready = false;
};
constexpr int kMaxDevices = 64;
DeviceScratch g_scratch[kMaxDevices];
std::mutex g_scratch_mu;

// Device addresses of the arrays above for the current device. Host code cannot use the
// array names as device addresses, so they are looked up once per device.
int scratch_for_current_device(DeviceScratch** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return EAGLE_ECUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  DeviceScratch& s = g_scratch[dev];
  if (!s.ready) {
    void* p = nullptr;
    void* t = nullptr;
    void* e = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_partials) != cudaSuccess) return EAGLE_ECUDA;
    if (cudaGetSymbolAddress(&t, g_noalloc_tickets) != cudaSuccess) return EAGLE_ECUDA;
    if (cudaGetSymbolAddress(&e, g_noalloc_status) != cudaSuccess) return EAGLE_ECUDA;
    // the status word starts at zero on every device (a blocking clear, once, at set-up)
    if (cudaMemset(e, 0, sizeof(g_noalloc_status)) != cudaSuccess) return EAGLE_ECUDA;
    s.partials = static_cast<float*>(p);
    s.tickets = static_cast<int*>(t);
    s.status = static_cast<int*>(e);
    s.ready = true;
  }
  *out = &s;
  return EAGLE_OK;
}

}  // namespace

extern "C" int eagle_op_gemm_noalloc(void* stream, const void* W, int N, int K, const void* X, int M, int epi,
                                     void* out, int ldo) {
  using namespace eagle;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (!W || !X || !out || M <= 0 || N <= 0 || K <= 0 || ldo < N || K % 8 || epi < 0 || epi > 2)
    return EAGLE_EINVAL;
  if (M > kNoallocMaxRows) return EAGLE_ECAPACITY;
  const int BN = gemm_bn_for(M);
  const long long tiles = (long long)((N + 127) / 128) * ((M + BN - 1) / BN);
  if (tiles > kNoallocMaxTiles) return EAGLE_ECAPACITY;
  DeviceScratch* s = nullptr;
  const int rc = scratch_for_current_device(&s);
  if (rc != EAGLE_OK) return rc;
  // the tickets must start at zero; a completed call leaves them at zero, but an
  // abandoned one (device timeout) may not, so clear the ones this call uses
  if (cudaMemsetAsync(s->tickets, 0, (size_t)tiles * sizeof(int), st) != cudaSuccess) return EAGLE_ECUDA;
  const int r = gemm_bf16(st, W, N, K, X, M, epi, out, ldo, s->partials,
                          sizeof(g_noalloc_partials) / sizeof(float), s->tickets, (int)tiles, s->status, nullptr,
                          /*cache_maps=*/false);
  return r == 0 ? EAGLE_OK : (r == -4 ? EAGLE_ECUDA : EAGLE_EINVAL);
}

extern "C" int eagle_op_gemm_noalloc_status(void* stream) {
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  DeviceScratch* s = nullptr;
  const int rc = scratch_for_current_device(&s);
  if (rc != EAGLE_OK) return rc;
  int h = 0;
  if (cudaMemcpyAsync(&h, s->status, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return EAGLE_ECUDA;
  if (h == 0) return EAGLE_OK;
  if (cudaMemsetAsync(s->status, 0, sizeof(int), st) != cudaSuccess || cudaStreamSynchronize(st) != cudaSuccess)
    return EAGLE_ECUDA;
  return h == DEVERR_MBAR_TIMEOUT ? EAGLE_ETIMEOUT : EAGLE_EDEVICE;
}
