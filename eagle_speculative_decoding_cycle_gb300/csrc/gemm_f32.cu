// fp32 SIMT GEMM for the fp32 model configuration, Y[M][N] = X[M][K] W[N][K]^T.
// A 1e-4 tolerance rules out TF32 tensor cores, so this path uses FFMA. Each output is
// accumulated over k in order, so results are deterministic.
#include "common.cuh"
#include "kernels.h"

namespace eagle {

constexpr int FT_M = 32, FT_N = 64, FT_K = 32;

__global__ void __launch_bounds__(256) gemm_f32_k(const float* __restrict__ W, int N, int K,
                                                  const float* __restrict__ X, int M, int epi,
                                                  float* __restrict__ out, int ldo) {
  PDL_ENTRY();
  __shared__ float xs[FT_M][FT_K + 1];
  __shared__ float ws[FT_N][FT_K + 1];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int m0 = blockIdx.y * FT_M, n0 = blockIdx.x * FT_N;
  float acc[2][4] = {};
  for (int k0 = 0; k0 < K; k0 += FT_K) {
    for (int i = threadIdx.x; i < FT_M * FT_K; i += 256) {
      const int r = i / FT_K, c = i % FT_K;
      xs[r][c] = (m0 + r < M && k0 + c < K) ? X[(size_t)(m0 + r) * K + k0 + c] : 0.f;
    }
    for (int i = threadIdx.x; i < FT_N * FT_K; i += 256) {
      const int r = i / FT_K, c = i % FT_K;
      ws[r][c] = (n0 + r < N && k0 + c < K) ? W[(size_t)(n0 + r) * K + k0 + c] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < FT_K; ++kk) {
      const float x0 = xs[ty * 2][kk], x1 = xs[ty * 2 + 1][kk];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float w = ws[tx + 16 * j][kk];
        acc[0][j] = fmaf(x0, w, acc[0][j]);
        acc[1][j] = fmaf(x1, w, acc[1][j]);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int m = m0 + ty * 2 + i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx + 16 * j;
      if (n >= N) continue;
      float* o = out + (size_t)m * ldo + n;
      if (epi == EPI_ADD_F32) *o += acc[i][j];
      else *o = acc[i][j];
    }
  }
}

int gemm_f32(cudaStream_t st, const float* W, int N, int K, const float* X, int M, int epi, float* out, int ldo) {
  if (M <= 0 || N <= 0 || K <= 0) return -1;
  if (epi != EPI_F32 && epi != EPI_ADD_F32) return -1;
  dim3 grid((N + FT_N - 1) / FT_N, (M + FT_M - 1) / FT_M);
  launch_k(gemm_f32_k, grid, 256, 0, st, W, N, K, X, M, epi, out, ldo);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace eagle
