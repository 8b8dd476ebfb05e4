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

// One CTA per row of NW warps: every thread folds the tile records t, t + 32 NW, ... (with
// 32 warps, launched for at most 1024 tiles, a single record per thread, already in rank
// order), each warp reduces its lanes, warp 0 reduces the warps. The warp count is a function of the
// vocabulary alone, so a row's result does not depend on how many rows are merged.
template <int NW>
__global__ void __launch_bounds__(NW * 32) head_merge_k(HeadParams p) {
  PDL_ENTRY();
  __shared__ float s_m[NW], s_s[NW], s_v[NW][16];
  __shared__ int s_i[NW][16];
  const int row = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = p.K;
  float lv[16], M, S;
  int li[16];
  if constexpr (NW == 32) {
#pragma unroll
    for (int k = 0; k < 16; ++k) { lv[k] = -INFINITY; li[k] = 0x7fffffff; }
    M = -INFINITY;
    S = 0.f;
    if ((int)threadIdx.x < p.n_tiles) {
      const float* rec = p.part + ((size_t)threadIdx.x * p.n_rows + row) * (2 + 2 * K);
      M = rec[0];
      S = M == -INFINITY ? 0.f : rec[1];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        if (k >= K) continue;
        const int id = __float_as_int(rec[3 + 2 * k]);
        if (id >= 0) { lv[k] = rec[2 + 2 * k]; li[k] = id; }
      }
    }
  } else {
    head_merge_fold(p, row, threadIdx.x, NW * 32, lv, li, M, S);
  }
  head_merge_warp(K, lv, li, M, S, lane, s_v[warp], s_i[warp]);
  if (lane == 0) { s_m[warp] = M; s_s[warp] = S; }
  __syncthreads();
  if (warp != 0) return;
  // lane w < NW holds warp w's sorted list
  for (int k = 0; k < 16; ++k) {
    lv[k] = (lane < NW && k < K) ? s_v[lane][k] : -INFINITY;
    li[k] = (lane < NW && k < K) ? s_i[lane][k] : 0x7fffffff;
  }
  M = lane < NW ? s_m[lane] : -INFINITY;
  S = lane < NW ? s_s[lane] : 0.f;
  __syncwarp();
  head_merge_warp(K, lv, li, M, S, lane, s_v[0], s_i[0]);   // warp 0's own slot, already read
  __syncwarp();
  if (lane < K) {
    p.top_id[row * K + lane] = s_i[0][lane] == 0x7fffffff ? -1 : s_i[0][lane];
    p.top_val[row * K + lane] = s_v[0][lane];
  }
  if (lane == 0) p.lse[row] = (M == -INFINITY) ? -INFINITY : M + logf(S);
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
  // up to 1024 tiles: one record per thread of a 32-warp CTA, launched without early start
  // (a 1024-thread CTA needs a whole SM's registers, so started early it only waits for the
  // LM-head GEMM's CTAs to leave; measured 0.14 ms per 8B batch-1 cycle faster this way);
  // more: 8 warps folding many
  if (p.n_tiles <= 1024) head_merge_k<32><<<p.n_rows, 1024, 0, st>>>(p);
  else launch_k(head_merge_k<8>, p.n_rows, 256, 0, st, p);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace eagle
