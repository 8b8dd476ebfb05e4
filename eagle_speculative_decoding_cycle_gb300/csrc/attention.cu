// Tree-masked attention over a KV cache.
//
// Each flattened tree row attends to the whole context plus the root and its own
// ancestors, never to a sibling branch ("EAGLE-2: Context-Aware Dynamic Draft Trees",
// section "The Mask Preserves Tree Semantics in One Target Pass", Figure 7). Row
// visibility of a key slot s:
//   causal mode: s <= row_slot (prefill, the drafter's context rows, plain decoding);
//   tree mode:   s < ctx_len, or s - ctx_len < T and bit (s - ctx_len) of the row's
//                ancestry bitmask is set (verify pass, drafter expansion rows).
// One CTA handles one KV head and a block of rows (all query heads of the GQA group),
// streams the KV slots in 32-key tiles through shared memory with coalesced loads, and
// keeps an online softmax per query vector (one warp per query vector group).
#include "common.cuh"
#include "kernels.h"

namespace eagle {

constexpr int QPW = 2;            // query vectors per warp
constexpr int AT_WARPS = 4;
constexpr int QV = QPW * AT_WARPS;
constexpr int KT = 32;            // keys per tile
constexpr int DMAX = 128;

template <typename T>
__global__ void __launch_bounds__(128) attn_simt_k(AttnArgs a) {
  __shared__ float sq[QV][DMAX];
  __shared__ float sk[KT][DMAX + 1];
  __shared__ float sv[KT][DMAX];
  const int G = a.nq / a.nkv;
  const int RB = QV / G;                       // rows per CTA
  const int nb = (a.rows_per_seq + RB - 1) / RB;
  const int kvh = blockIdx.x;
  const int sidx = blockIdx.y / nb, rb = blockIdx.y % nb;
  const int r0 = sidx * a.rows_per_seq + rb * RB;
  const int r1 = min(r0 + RB, min((sidx + 1) * a.rows_per_seq, a.R));
  if (r0 >= r1) return;
  const int seq = a.row_seq[r0];
  const int d = a.d;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const T* qp = reinterpret_cast<const T*>(a.q);
  const T* kc = reinterpret_cast<const T*>(a.kcache) + (size_t)(seq * a.nkv + kvh) * a.cap * d;
  const T* vc = reinterpret_cast<const T*>(a.vcache) + (size_t)(seq * a.nkv + kvh) * a.cap * d;
  const int ctx = a.ctx_len[seq];

  // load the query vectors: qv = (row - r0) * G + g
  for (int i = threadIdx.x; i < QV * d; i += blockDim.x) {
    const int qv = i / d, c = i % d;
    const int r = r0 + qv / G;
    sq[qv][c] = (r < r1) ? Elem<T>::to_f(qp[((size_t)r * a.nq + kvh * G + qv % G) * d + c]) : 0.f;
  }
  int kend = 0;
  for (int r = r0; r < r1; ++r) {
    const int e = a.mode == 0 ? a.row_slot[r] + 1 : ctx + a.tree_T;
    kend = max(kend, e);
  }
  kend = min(kend, a.cap);

  float m[QPW], l[QPW], o[QPW][DMAX / 32];
#pragma unroll
  for (int j = 0; j < QPW; ++j) {
    m[j] = -INFINITY;
    l[j] = 0.f;
#pragma unroll
    for (int c = 0; c < DMAX / 32; ++c) o[j][c] = 0.f;
  }
  for (int t0 = 0; t0 < kend; t0 += KT) {
    __syncthreads();
    for (int i = threadIdx.x; i < KT * d; i += blockDim.x) {
      const int kk = i / d, c = i % d;
      const int s = t0 + kk;
      const bool in = s < kend;
      sk[kk][c] = in ? Elem<T>::to_f(kc[(size_t)s * d + c]) : 0.f;
      sv[kk][c] = in ? Elem<T>::to_f(vc[(size_t)s * d + c]) : 0.f;
    }
    __syncthreads();
    const int s = t0 + lane;
#pragma unroll
    for (int j = 0; j < QPW; ++j) {
      const int qv = warp * QPW + j;
      const int r = r0 + qv / G;
      if (r >= r1) continue;
      bool vis;
      if (a.mode == 0) {
        vis = s <= a.row_slot[r];
      } else {
        const int t = s - ctx;
        vis = s < ctx || (t >= 0 && t < a.tree_T &&
                          ((a.mask[(size_t)r * a.mask_words + (t >> 6)] >> (t & 63)) & 1ull));
      }
      vis = vis && s < kend;
      float sc = -INFINITY;
      if (vis) {
        float acc = 0.f;
        for (int c = 0; c < d; ++c) acc += sq[qv][c] * sk[lane][c];
        sc = acc * a.scale;
      }
      const float mt = warp_max(sc);
      const float mn = fmaxf(m[j], mt);
      if (mn == -INFINITY) continue;
      const float p = vis ? expf(sc - mn) : 0.f;
      const float corr = expf(m[j] - mn);
      l[j] = l[j] * corr + warp_sum(p);
      m[j] = mn;
#pragma unroll
      for (int c = 0; c < DMAX / 32; ++c) o[j][c] *= corr;
      for (int kk = 0; kk < KT; ++kk) {
        const float pk = __shfl_sync(0xffffffffu, p, kk);
        if (pk != 0.f) {
#pragma unroll
          for (int c = 0; c < DMAX / 32; ++c) {
            const int dim = lane + 32 * c;
            if (dim < d) o[j][c] += pk * sv[kk][dim];
          }
        }
      }
    }
  }
  T* op = reinterpret_cast<T*>(a.out);
#pragma unroll
  for (int j = 0; j < QPW; ++j) {
    const int qv = warp * QPW + j;
    const int r = r0 + qv / G;
    if (r >= r1) continue;
    const float inv = l[j] > 0.f ? 1.f / l[j] : 0.f;
#pragma unroll
    for (int c = 0; c < DMAX / 32; ++c) {
      const int dim = lane + 32 * c;
      if (dim < d) op[((size_t)r * a.nq + kvh * G + qv % G) * d + dim] = Elem<T>::from_f(o[j][c] * inv);
    }
  }
}

int attention(cudaStream_t st, int dtype, const AttnArgs& a) {
  if (a.R <= 0) return 0;
  if (a.d > DMAX || a.nq % a.nkv) return -1;
  const int G = a.nq / a.nkv;
  if (G > QV || QV % G) return -1;
  const int RB = QV / G;
  const int nseq = (a.R + a.rows_per_seq - 1) / a.rows_per_seq;
  const int nb = (a.rows_per_seq + RB - 1) / RB;
  dim3 grid(a.nkv, nseq * nb);
  if (dtype == DT_F32) attn_simt_k<float><<<grid, 128, 0, st>>>(a);
  else attn_simt_k<__nv_bfloat16><<<grid, 128, 0, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace eagle
