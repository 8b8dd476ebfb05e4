// LM-head reductions outside the GEMM: partial records from materialised logits (fp32
// model path) and the fixed-order merge of the per-tile records into per-row top-K and
// log-sum-exp (both paths).
#include "common.cuh"
#include "kernels.h"
#include "lmhead.cuh"

namespace eagle {

constexpr int HP_ROWS = 8;

__global__ void __launch_bounds__(128) head_partials_k(const float* logits, int ld, HeadParams p) {
  PDL_ENTRY();
  __shared__ float vals[HP_ROWS][128];
  const int tile = blockIdx.x;
  const int r0 = blockIdx.y * HP_ROWS;
  for (int i = threadIdx.x; i < HP_ROWS * 128; i += 128) {
    const int rr = i / 128, c = i % 128;
    const int r = r0 + rr, v = tile * 128 + c;
    vals[rr][c] = (r < p.n_rows && v < p.vocab) ? logits[(size_t)r * ld + v] : 0.f;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int rr = warp; rr < HP_ROWS; rr += 4) {
    const int r = r0 + rr;
    if (r < p.n_rows) head_tile_row(vals[rr], tile, r, p, lane);
  }
}

__global__ void __launch_bounds__(128) head_merge_k(HeadParams p) {
  PDL_ENTRY();
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (row < p.n_rows) head_merge_row(p, row, threadIdx.x & 31);
}

size_t head_part_bytes(int vocab, int rows, int K) {
  return (size_t)((vocab + 127) / 128) * rows * (2 + 2 * K) * sizeof(float);
}

int head_partials_from_logits(cudaStream_t st, const float* logits, int ld, const HeadParams& p) {
  if (p.n_rows <= 0) return 0;
  if (p.K < 1 || p.K > 16) return -1;
  dim3 grid(p.n_tiles, (p.n_rows + HP_ROWS - 1) / HP_ROWS);
  launch_k(head_partials_k, grid, 128, 0, st, logits, ld, p);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

int head_merge(cudaStream_t st, const HeadParams& p) {
  if (p.n_rows <= 0) return 0;
  if (p.K < 1 || p.K > 16) return -1;
  launch_k(head_merge_k, (p.n_rows + 3) / 4, 128, 0, st, p);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace eagle
