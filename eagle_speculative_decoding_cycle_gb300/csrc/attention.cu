// Tree-masked attention over a KV cache.
//
// Each flattened tree row attends to the whole context plus the root and its own
// ancestors, never to a sibling branch ("EAGLE-2: Context-Aware Dynamic Draft Trees",
// section "The Mask Preserves Tree Semantics in One Target Pass", Figure 7). Row
// visibility of a key slot s:
//   causal mode: s <= row_slot (prefill, the drafter's context rows, plain decoding);
//   training-time-test mode (the EAGLE-3 multi-step drafter pass), n = ctx_len: a row at
//     slot < n is causal; a row at slot n(j-1) + t (step j >= 2 of source t) sees slots
//     0..t and its own source's earlier steps n(i-1) + t, i = 2..j;
//   tree mode:   s < ctx_len, or s - ctx_len < T and bit (s - ctx_len) of the row's
//                ancestry bitmask is set (verify pass, drafter expansion rows).
// One CTA handles one KV head and a block of rows (all query heads of the GQA group),
// streams the KV slots in 32-key tiles through shared memory with coalesced loads, and
// keeps an online softmax per query vector (one warp per query vector group).
#include "common.cuh"
#include "kernels.h"

#include <algorithm>

namespace eagle {

constexpr int QPW = 2;            // query vectors per warp
constexpr int AT_WARPS = 4;
constexpr int QV = QPW * AT_WARPS;
constexpr int KT = 32;            // keys per tile
constexpr int DMAX = 128;

// training-time-test visibility of key slot `key` for a row at `slot`, n = sequence length
__device__ __forceinline__ bool ttt_visible(int slot, int key, int n) {
  if (slot < n) return key <= slot;
  const int t = slot % n;
  return key < n ? key <= t : ((key - n) % n == t && key <= slot);
}


template <typename T>
__global__ void __launch_bounds__(128) attn_simt_k(AttnArgs a) {
  PDL_ENTRY();
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
  const T* kc = reinterpret_cast<const T*>(a.kcache);
  const T* vc = reinterpret_cast<const T*>(a.vcache);
  const int ctx = a.ctx_len[seq];

  // load the query vectors: qv = (row - r0) * G + g
  for (int i = threadIdx.x; i < QV * d; i += blockDim.x) {
    const int qv = i / d, c = i % d;
    const int r = r0 + qv / G;
    sq[qv][c] = (r < r1) ? Elem<T>::to_f(qp[((size_t)r * a.nq + kvh * G + qv % G) * d + c]) : 0.f;
  }
  int kend = 0;
  for (int r = r0; r < r1; ++r) {
    const int e = a.mode == 1 ? ctx + a.tree_T : a.row_slot[r] + 1;
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
      const size_t ro = in ? kv_row(a.page, seq, a.nkv, kvh, a.cap, s) * d + c : 0;
      sk[kk][c] = in ? Elem<T>::to_f(kc[ro]) : 0.f;
      sv[kk][c] = in ? Elem<T>::to_f(vc[ro]) : 0.f;
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
      } else if (a.mode == 2) {
        vis = ttt_visible(a.row_slot[r], s, ctx);
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

int attention_bf16_mma(cudaStream_t st, const AttnArgs& a);

int attention(cudaStream_t st, int dtype, const AttnArgs& a) {
  if (a.R <= 0) return 0;
  if (dtype == DT_BF16) return attention_bf16_mma(st, a);
  if (a.d > DMAX || a.nq % a.nkv) return -1;
  const int G = a.nq / a.nkv;
  if (G > QV || QV % G) return -1;
  const int RB = QV / G;
  const int nseq = (a.R + a.rows_per_seq - 1) / a.rows_per_seq;
  const int nb = (a.rows_per_seq + RB - 1) / RB;
  dim3 grid(a.nkv, nseq * nb);
  if (dtype == DT_F32) launch_k(attn_simt_k<float>, grid, 128, 0, st, a);
  else launch_k(attn_simt_k<__nv_bfloat16>, grid, 128, 0, st, a);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace eagle

// ------------------------------------------------------------------------------------------------
// Tensor-core path (bf16): mma.sync m16n8k16 with fp32 accumulation, FlashAttention-style
// online softmax in the exp2 domain, K/V tiles of 64 keys double-buffered in shared memory
// by cp.async, and split-KV over the key range with a fixed-order log-sum-exp combine.
// A CTA covers one KV head and 64 query vectors (rows x the GQA group); warp w owns query
// vectors 16w .. 16w+15.
// ------------------------------------------------------------------------------------------------
namespace eagle {

constexpr int MT_KEYS = 64;
constexpr int MT_QV = 64;

__device__ __forceinline__ void mma_bf16_16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// (lo, hi) -> bf16 pairs of their high parts and of the residuals x - bf16(x).
__device__ __forceinline__ void split_bf16(float lo, float hi, uint32_t& h, uint32_t& l) {
  const __nv_bfloat162 hv = __floats2bfloat162_rn(lo, hi);
  const float2 back = __bfloat1622float2(hv);
  const __nv_bfloat162 lv = __floats2bfloat162_rn(lo - back.x, hi - back.y);
  h = *reinterpret_cast<const uint32_t*>(&hv);
  l = *reinterpret_cast<const uint32_t*>(&lv);
}

// a row's visibility data: validity, own slot, and (tree mode) the 64 mask bits of the
// current key tile, bit i <-> key tile_base + i
struct RowVis {
  int valid, slot;
  uint64_t win;
};

// Bits [base, base + 64) of a row's tree mask (4 words in shared memory); bits below 0 and
// past the words read as 0.
__device__ __forceinline__ uint64_t mask_window(const uint64_t* mw, int base) {
  if (base <= -64 || base >= 256) return 0ull;
  if (base < 0) return mw[0] << (-base);
  const int w = base >> 6, sh = base & 63;
  const uint64_t lo = mw[w] >> sh;
  const uint64_t hi = (sh && w < 3) ? mw[w + 1] << (64 - sh) : 0ull;
  return lo | hi;
}

template <bool TTT>
__device__ __forceinline__ bool visible(const AttnArgs& a, const RowVis& rv, int ctx, int key, int kb) {
  if (!rv.valid) return false;
  if constexpr (TTT) return ttt_visible(rv.slot, key, ctx);
  if (a.mode == 0) return key <= rv.slot;
  if (key < ctx) return true;
  if (key - ctx >= a.tree_T) return false;
  return (rv.win >> (key - kb)) & 1ull;
}

// Everything before the query loads reads data older than the preceding kernel (the rows'
// sequence, slot, mask and context length, and in tree mode the context keys below
// ctx_len, which that kernel never writes), so it runs before waiting on that kernel: the
// first key tile of a tree-mode CTA is already in flight when the queries arrive.
// KIND: 0 = contiguous cache, 1 = paged cache, 2 = training-time-test mask (contiguous);
// one instantiation each, so the cycle's contiguous kernel carries neither of the others.
template <int D, int KIND>
__global__ void __launch_bounds__(128, 3) attn_mma_k(AttnArgs a, int splits) {
  constexpr int LD = D + 8;                      // padded smem row (bf16 elements)
  extern __shared__ __align__(16) uint8_t attn_smem[];
  __nv_bfloat16* sK = reinterpret_cast<__nv_bfloat16*>(attn_smem);              // [2][64][LD]
  __nv_bfloat16* sV = sK + 2 * MT_KEYS * LD;                                    // [2][64][LD]
  const int G = a.nq / a.nkv;
  const int RB = MT_QV / G;
  const int nb = (a.rows_per_seq + RB - 1) / RB;
  const int kvh = blockIdx.x;
  const int sidx = blockIdx.y / nb, rb = blockIdx.y % nb;
  const int split = blockIdx.z;
  const int r0 = sidx * a.rows_per_seq + rb * RB;
  const int r1 = min(r0 + RB, min((sidx + 1) * a.rows_per_seq, a.R));
  if (r0 >= r1) return;
  const int seq = a.row_seq[r0];
  const int ctx = a.ctx_len[seq];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const __nv_bfloat16* kc = reinterpret_cast<const __nv_bfloat16*>(a.kcache);
  const __nv_bfloat16* vc = reinterpret_cast<const __nv_bfloat16*>(a.vcache);

  int kend = 0;
  for (int r = r0; r < r1; ++r) kend = max(kend, a.mode == 1 ? ctx + a.tree_T : a.row_slot[r] + 1);
  kend = min(kend, a.cap);
  const int n_tiles = (kend + MT_KEYS - 1) / MT_KEYS;
  const int tps = (n_tiles + splits - 1) / splits;
  const int t_begin = split * tps, t_end = min(n_tiles, t_begin + tps);

  // the two query vectors (rows of the mma fragment) this thread holds
  const int qv_a = warp * 16 + (lane >> 2), qv_b = qv_a + 8;
  RowVis va, vb;
  auto setup_row = [&](int qv, RowVis& v, int& row, int& head) {
    row = r0 + qv / G;
    head = kvh * G + qv % G;
    v.valid = row < r1;
    v.slot = v.valid ? a.row_slot[row] : -1;
    v.win = 0ull;
  };
  int row_a, head_a, row_b, head_b;
  setup_row(qv_a, va, row_a, head_a);
  setup_row(qv_b, vb, row_b, head_b);

  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;
  const float sl2 = a.scale * 1.4426950408889634f;

  // contiguous cache: one (sequence, head) run of rows; paged: rows through the block table
  const size_t head_row0 = KIND == 1 ? 0 : ((size_t)seq * a.nkv + kvh) * (size_t)a.cap;
  auto load_tile = [&](int t, int buf) {
    constexpr int CH = D / 8;   // 16-byte chunks per row
    for (int i = threadIdx.x; i < MT_KEYS * CH; i += 128) {
      const int kr = i / CH, c = i % CH;
      const int key = t * MT_KEYS + kr;
      const bool in = key < kend;
      const int kk = in ? key : 0;
      size_t grow;
      if constexpr (KIND == 1) grow = kv_row(a.page, seq, a.nkv, kvh, a.cap, kk);
      else grow = head_row0 + kk;
      const size_t goff = grow * D + c * 8;
      const uint32_t dk = smem_u32(sK + (buf * MT_KEYS + kr) * LD + c * 8);
      const uint32_t dv = smem_u32(sV + (buf * MT_KEYS + kr) * LD + c * 8);
      cp_async16(dk, kc + goff, in ? 16 : 0);
      cp_async16(dv, vc + goff, in ? 16 : 0);
    }
    cp_async_commit();
  };

  // the block's rows' tree masks, [row in block][4 words]
  __shared__ uint64_t s_mask[MT_QV][4];
  if (a.mode == 1) {
    for (int i = threadIdx.x; i < RB * 4; i += 128) {
      const int rr = i >> 2, w = i & 3, row = r0 + rr;
      s_mask[rr][w] = (row < r1 && w < a.mask_words) ? a.mask[(size_t)row * a.mask_words + w] : 0ull;
    }
  }
  const bool early = a.mode == 1 && t_begin < t_end && (t_begin + 1) * MT_KEYS <= ctx;
  if (early) load_tile(t_begin, 0);
  PDL_ENTRY();
  // Q fragments (bf16 pairs), zero for rows past the block
  uint32_t qf[D / 16][4];
  {
    const __nv_bfloat16* qp = reinterpret_cast<const __nv_bfloat16*>(a.q);
    const __nv_bfloat16* pa = qp + ((size_t)row_a * a.nq + head_a) * D;
    const __nv_bfloat16* pb = qp + ((size_t)row_b * a.nq + head_b) * D;
    const int c = (lane & 3) * 2;
#pragma unroll
    for (int kt = 0; kt < D / 16; ++kt) {
      qf[kt][0] = va.valid ? *reinterpret_cast<const uint32_t*>(pa + kt * 16 + c) : 0u;
      qf[kt][1] = vb.valid ? *reinterpret_cast<const uint32_t*>(pb + kt * 16 + c) : 0u;
      qf[kt][2] = va.valid ? *reinterpret_cast<const uint32_t*>(pa + kt * 16 + 8 + c) : 0u;
      qf[kt][3] = vb.valid ? *reinterpret_cast<const uint32_t*>(pb + kt * 16 + 8 + c) : 0u;
    }
  }
  if (!early && t_begin < t_end) load_tile(t_begin, 0);
  const bool warp_live = warp * 16 < (r1 - r0) * G;
  for (int t = t_begin; t < t_end; ++t) {
    const int buf = (t - t_begin) & 1;
    if (t + 1 < t_end) { load_tile(t + 1, buf ^ 1); cp_async_wait<1>(); }
    else cp_async_wait<0>();
    __syncthreads();
    const int kb = t * MT_KEYS;
    // a warp whose 16 query vectors are all past the block's rows only helps load the tiles
    if (!warp_live) { __syncthreads(); continue; }
    if (a.mode == 1 && kb + MT_KEYS > ctx) {   // the tile reaches the tree rows' keys
      va.win = va.valid ? mask_window(s_mask[row_a - r0], kb - ctx) : 0ull;
      vb.win = vb.valid ? mask_window(s_mask[row_b - r0], kb - ctx) : 0ull;
    }
    const __nv_bfloat16* K = sK + buf * MT_KEYS * LD;
    const __nv_bfloat16* Vt = sV + buf * MT_KEYS * LD;
    float s[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
      const __nv_bfloat16* kr = K + (nt * 8 + (lane >> 2)) * LD + (lane & 3) * 2;
#pragma unroll
      for (int kt = 0; kt < D / 16; ++kt) {
        const uint32_t b0 = *reinterpret_cast<const uint32_t*>(kr + kt * 16);
        const uint32_t b1 = *reinterpret_cast<const uint32_t*>(kr + kt * 16 + 8);
        mma_bf16_16816(s[nt], qf[kt], b0, b1);
      }
    }
    // mask, scale to the exp2 domain, running max
    float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int key = t * MT_KEYS + nt * 8 + (lane & 3) * 2 + e;
        s[nt][e] = visible<KIND == 2>(a, va, ctx, key, kb) ? s[nt][e] * sl2 : -INFINITY;
        s[nt][2 + e] = visible<KIND == 2>(a, vb, ctx, key, kb) ? s[nt][2 + e] * sl2 : -INFINITY;
        mx_a = fmaxf(mx_a, s[nt][e]);
        mx_b = fmaxf(mx_b, s[nt][2 + e]);
      }
    }
    mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
    mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
    mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
    mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
    const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
    const float base_a = mn_a == -INFINITY ? 0.f : mn_a, base_b = mn_b == -INFINITY ? 0.f : mn_b;
    const float corr_a = exp2f(m_a - base_a), corr_b = exp2f(m_b - base_b);
    m_a = mn_a;
    m_b = mn_b;
    float ps_a = 0.f, ps_b = 0.f;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      s[nt][0] = exp2f(s[nt][0] - base_a);
      s[nt][1] = exp2f(s[nt][1] - base_a);
      s[nt][2] = exp2f(s[nt][2] - base_b);
      s[nt][3] = exp2f(s[nt][3] - base_b);
      ps_a += s[nt][0] + s[nt][1];
      ps_b += s[nt][2] + s[nt][3];
    }
    l_a = l_a * corr_a + ps_a;
    l_b = l_b * corr_b + ps_b;
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
      o[i][0] *= corr_a; o[i][1] *= corr_a;
      o[i][2] *= corr_b; o[i][3] *= corr_b;
    }
    // O += P V. P is split into a bf16 high part and a bf16 residual so that the product
    // carries ~16 bits of P (a single bf16 P would perturb every attention output by up to
    // 2^-9 relative, an error that then accumulates across the layers).
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t ph[4], pl[4];
      split_bf16(s[2 * kk][0], s[2 * kk][1], ph[0], pl[0]);
      split_bf16(s[2 * kk][2], s[2 * kk][3], ph[1], pl[1]);
      split_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1], ph[2], pl[2]);
      split_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3], ph[3], pl[3]);
      const int mi = lane >> 3;
      const int key = kk * 16 + (mi & 1) * 8 + (lane & 7);
#pragma unroll
      for (int dp = 0; dp < D / 16; ++dp) {
        uint32_t b[4];
        ldsm_x4_trans(smem_u32(Vt + key * LD + dp * 16 + (mi >> 1) * 8), b);
        mma_bf16_16816(o[2 * dp], ph, b[0], b[1]);
        mma_bf16_16816(o[2 * dp + 1], ph, b[2], b[3]);
        mma_bf16_16816(o[2 * dp], pl, b[0], b[1]);
        mma_bf16_16816(o[2 * dp + 1], pl, b[2], b[3]);
      }
    }
    __syncthreads();
  }
  l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
  l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
  const int c = (lane & 3) * 2;
  if (splits == 1) {
    __nv_bfloat16* op = reinterpret_cast<__nv_bfloat16*>(a.out);
    const float ia = l_a > 0.f ? 1.f / l_a : 0.f, ib = l_b > 0.f ? 1.f / l_b : 0.f;
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
      if (va.valid)
        *reinterpret_cast<__nv_bfloat162*>(op + ((size_t)row_a * a.nq + head_a) * D + i * 8 + c) =
            __floats2bfloat162_rn(o[i][0] * ia, o[i][1] * ia);
      if (vb.valid)
        *reinterpret_cast<__nv_bfloat162*>(op + ((size_t)row_b * a.nq + head_b) * D + i * 8 + c) =
            __floats2bfloat162_rn(o[i][2] * ib, o[i][3] * ib);
    }
  } else {
    const size_t sa = ((size_t)split * a.R + row_a) * a.nq + head_a;
    const size_t sb = ((size_t)split * a.R + row_b) * a.nq + head_b;
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
      if (va.valid) *reinterpret_cast<float2*>(a.part_o + sa * D + i * 8 + c) = make_float2(o[i][0], o[i][1]);
      if (vb.valid) *reinterpret_cast<float2*>(a.part_o + sb * D + i * 8 + c) = make_float2(o[i][2], o[i][3]);
    }
    if ((lane & 3) == 0) {
      if (va.valid) { a.part_ml[sa * 2] = m_a; a.part_ml[sa * 2 + 1] = l_a; }
      if (vb.valid) { a.part_ml[sb * 2] = m_b; a.part_ml[sb * 2 + 1] = l_b; }
    }
  }
}

// out[r][h] = sum_s o_s 2^(m_s - M) / sum_s l_s 2^(m_s - M), splits in order. One warp per
// (row, head): lane s holds split s's (m, l); every split's partial output is loaded before
// the in-order sums, so the kernel costs two dependent loads instead of one per split.
constexpr int MAX_SPLITS = 16;
template <int D>
__global__ void attn_combine_k(AttnArgs a, int splits) {
  PDL_ENTRY();
  const int qi = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (qi >= a.R * a.nq) return;
  const size_t stride = (size_t)a.R * a.nq;
  float ms = -INFINITY, ls = 0.f;
  if (lane < splits) {
    ms = a.part_ml[((size_t)lane * stride + qi) * 2];
    ls = a.part_ml[((size_t)lane * stride + qi) * 2 + 1];
  }
  float x[MAX_SPLITS][D / 32];
#pragma unroll
  for (int sp = 0; sp < MAX_SPLITS; ++sp)
#pragma unroll
    for (int i = 0; i < D / 32; ++i)
      x[sp][i] = sp < splits ? a.part_o[((size_t)sp * stride + qi) * D + lane + 32 * i] : 0.f;
  float M = ms;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const float w = ms == -INFINITY ? 0.f : exp2f(ms - M);
  float L = 0.f;
  float acc[D / 32];
#pragma unroll
  for (int i = 0; i < D / 32; ++i) acc[i] = 0.f;
#pragma unroll
  for (int sp = 0; sp < MAX_SPLITS; ++sp) {
    const float ws = __shfl_sync(0xffffffffu, w, sp);
    const float lw = __shfl_sync(0xffffffffu, ls * w, sp);
    const float msp = __shfl_sync(0xffffffffu, ms, sp);
    if (sp < splits && msp != -INFINITY) {
      L += lw;
#pragma unroll
      for (int i = 0; i < D / 32; ++i) acc[i] += x[sp][i] * ws;
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  __nv_bfloat16* op = reinterpret_cast<__nv_bfloat16*>(a.out);
#pragma unroll
  for (int i = 0; i < D / 32; ++i) op[(size_t)qi * D + lane + 32 * i] = __float2bfloat16_rn(acc[i] * inv);
}

size_t attention_scratch_floats(int rows, int nq, int d) { return (size_t)16 * rows * nq * (d + 2); }

template <int D>
static int launch_mma(cudaStream_t st, const AttnArgs& a) {
  const int G = a.nq / a.nkv;
  const int RB = MT_QV / G;
  const int nseq = (a.R + a.rows_per_seq - 1) / a.rows_per_seq;
  const int nb = (a.rows_per_seq + RB - 1) / RB;
  const int base = a.nkv * nseq * nb;
  const size_t smem = (size_t)4 * MT_KEYS * (D + 8) * sizeof(__nv_bfloat16);
  static int sms = 0, per_sm = 1;
  if (!sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaFuncSetAttribute(attn_mma_k<D, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    cudaFuncSetAttribute(attn_mma_k<D, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    cudaFuncSetAttribute(attn_mma_k<D, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attn_mma_k<D, 0>, 128, smem) != cudaSuccess ||
        per_sm < 1)
      per_sm = 1;
  }
  // as many key splits as one wave of resident CTAs holds (a second, partial wave would
  // double the time of this latency-bound kernel)
  int splits = per_sm * sms / base;
  const int max_tiles = (a.cap + MT_KEYS - 1) / MT_KEYS;
  splits = std::min(std::min(splits, MAX_SPLITS), max_tiles);
  while (splits > 1 && (size_t)splits * a.R * a.nq * D > a.part_floats) --splits;
  if (!a.part_o || !a.part_ml) splits = 1;
  if (splits < 1) splits = 1;
  // the training-time-test mask is its own instantiation, so the cycle's kernel stays lean
  const dim3 grid(a.nkv, nseq * nb, splits);
  if (a.mode == 2 && !a.page.table) launch_k(attn_mma_k<D, 2>, grid, 128, smem, st, a, splits);
  else if (a.mode == 2) return -1;   // the training-time test runs on the contiguous drafter cache
  else if (a.page.table) launch_k(attn_mma_k<D, 1>, grid, 128, smem, st, a, splits);
  else launch_k(attn_mma_k<D, 0>, grid, 128, smem, st, a, splits);
  if (splits > 1) launch_k(attn_combine_k<D>, (a.R * a.nq + 3) / 4, 128, 0, st, a, splits);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

int attention_bf16_mma(cudaStream_t st, const AttnArgs& a) {
  const int G = a.nq / a.nkv;
  if (G < 1 || G > MT_QV || MT_QV % G) return -1;
  if (a.mode == 1 && (a.mask_words > 4 || a.tree_T > 256)) return -1;
  switch (a.d) {
    case 32: return launch_mma<32>(st, a);
    case 64: return launch_mma<64>(st, a);
    case 128: return launch_mma<128>(st, a);
  }
  return -1;
}

}  // namespace eagle
