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
#include "tc_common.cuh"

#include <algorithm>
#include <cstdlib>
#include <cstring>

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
// Tensor-core path (bf16), with a result for each query row that does not depend on which
// other rows share the launch.
//
// A row at logical position P attends to the keys of positions 0..P: positions below the
// context length are the cache slots of the same number; a tree row's positions from the
// context length on are its ancestors (the root, ..., itself), one per depth, whose slots
// are the set bits of its ancestry mask in increasing order (generation order is depth
// major, so an ancestor always precedes its descendants); a training-time-test row of step
// j >= 2 and source t reads positions t+1 .. t+j-1 from its own source chain. The softmax
// over those keys is computed in a fixed decomposition that depends on P alone:
//   body  -- positions [0, B) with B = min(P + 1 - TAIL_MIN, first non-plain position),
//            in fixed key splits of `tps` 64-key tiles (split s: tiles s*tps ..), each an
//            online softmax over its tiles in order on the tensor cores (mma.sync
//            m16n8k16, fp32 accumulation, P split into bf16 high and residual parts);
//   tail  -- positions [B, P] (TAIL_MIN keys, or fewer near the start), one FFMA pass in
//            position order;
//   merge -- the body splits in order, then the tail, by log-sum-exp weights.
// The body splits and the tail run as CTAs of one launch (the tail needs no body result),
// each leaving an (m, l, o) partial; a second launch merges a row's partials in order.
// The split length `tps` is a function of the cache capacity, the engine's batch capacity and
// the scratch size only, so a verify row and the plain-decoding step at the same position go
// through the same arithmetic and give bit-identical outputs (greedy speculative decoding then
// reproduces the GPU's own plain decoding exactly, "EAGLE: Feature-Level Drafting",
// "Speculative decoding in four moves", item 4). With head dim 128 the bodies can instead run
// on tcgen05 (attn_tc_k below, EAGLE_ATTN_TC=1 for the whole process).
// ------------------------------------------------------------------------------------------------
namespace eagle {

constexpr int MT_KEYS = 64;       // keys per body tile
constexpr int TAIL_MIN = 16;      // the last TAIL_MIN positions of a row form its tail
constexpr int MAX_SPLITS = 31;    // body splits; with the tail, one partial per lane of the merge
constexpr int TAIL_ITEMS = 8;     // (row, query head) items per tail CTA, two per warp

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

// (lo, hi) -> bf16 pairs of their high parts and of the residuals x - bf16(x).
__device__ __forceinline__ void split_bf16(float lo, float hi, uint32_t& h, uint32_t& l) {
  const __nv_bfloat162 hv = __floats2bfloat162_rn(lo, hi);
  const float2 back = __bfloat1622float2(hv);
  const __nv_bfloat162 lv = __floats2bfloat162_rn(lo - back.x, hi - back.y);
  h = *reinterpret_cast<const uint32_t*>(&hv);
  l = *reinterpret_cast<const uint32_t*>(&lv);
}

// A row's logical position P, the end of its plain-slot prefix (positions p < plain_end sit
// at slot p), and the end of its body.
struct RowSpan {
  int P, plain_end, body;
};

__device__ __forceinline__ RowSpan row_span(const AttnArgs& a, int r, int ctx) {
  RowSpan s;
  const int slot = a.row_slot[r];
  if (a.mode == 1) {
    int c = 0;
    for (int w = 0; w < a.mask_words; ++w) c += __popcll(a.mask[(size_t)r * a.mask_words + w]);
    s.P = ctx + c - 1;
    s.plain_end = ctx;
  } else if (a.mode == 2 && ctx > 0 && slot >= ctx) {
    const int t = slot % ctx;
    s.P = t + slot / ctx;
    s.plain_end = t + 1;
  } else {
    s.P = slot;
    s.plain_end = slot + 1;
  }
  s.body = max(0, min(s.P + 1 - TAIL_MIN, s.plain_end));
  return s;
}

// Tail of up to TAIL_ITEMS (row, query head) items of a row block: stages the plain slots of
// their tails (positions [min body, max plain tail end)) and, in tree mode, the T tree slots;
// then each warp takes two items: the scores in position order (four lanes per key, a
// quarter of the head dimension each, summed (q0 + q1) + (q2 + q3)), their softmax, and P.V in
// position order, written as the row's partial after its body splits. Training-time-test
// chain keys are read from the cache directly.
template <int D, int KIND, int ITEMS = TAIL_ITEMS>
__device__ __forceinline__ void tail_chunk(const AttnArgs& a, int tps, int r0, int r1, int kvh, int chunk, int nB,
                                           int tail_cap, uint8_t* smem) {
  constexpr int LD = D + 8;
  constexpr int DL = D / 32;                         // output dims per lane
  constexpr int DQ = D / 4;                          // score dims per lane (a quarter)
  __shared__ int s_P[ITEMS], s_pe[ITEMS], s_body[ITEMS];
  __shared__ int s_lo, s_hi;
  const int G = a.nq / a.nkv;
  const int it0 = chunk * ITEMS;
  const int n_items = min(ITEMS, (r1 - r0) * G - it0);
  if (n_items <= 0) return;
  const int ra = r0 + it0 / G, rz = r0 + (it0 + n_items - 1) / G;   // rows [ra, rz]
  const int nA_cap = TAIL_MIN + ITEMS;
  __nv_bfloat16* sAK = reinterpret_cast<__nv_bfloat16*>(smem);
  __nv_bfloat16* sAV = sAK + (size_t)nA_cap * LD;
  __nv_bfloat16* sBK = sAV + (size_t)nA_cap * LD;
  __nv_bfloat16* sBV = sBK + (size_t)nB * LD;
  uint8_t* wbase = reinterpret_cast<uint8_t*>(sBV + (size_t)nB * LD);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int seq = a.row_seq[r0];
  const int ctx = a.ctx_len[seq];
  if (threadIdx.x <= rz - ra) {
    const RowSpan rs = row_span(a, ra + threadIdx.x, ctx);
    s_P[threadIdx.x] = rs.P;
    s_pe[threadIdx.x] = rs.plain_end;
    s_body[threadIdx.x] = rs.body;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int lo = INT32_MAX, hi = 0;
    for (int i = 0; i <= rz - ra; ++i) {
      lo = min(lo, s_body[i]);
      hi = max(hi, min(s_P[i] + 1, s_pe[i]));
    }
    if (hi < lo) hi = lo;
    if (hi - lo > nA_cap) { latch_error(a.err, DEVERR_BOUNDS); hi = lo; lo = -1; }
    s_lo = lo;
    s_hi = hi;
  }
  // The query vectors and the tree rows' keys come from the preceding kernel. In tree mode the
  // plain tail keys are context (slots below ctx_len, which that kernel does not write): they
  // are staged before the wait.
  const bool pre = a.mode == 1;
  if (pre) {
    __syncthreads();
  } else {
    PDL_ENTRY();
    __syncthreads();
  }
  if (s_lo < 0) return;
  const int lo = s_lo, nA = s_hi - s_lo;
  const __nv_bfloat16* kc = reinterpret_cast<const __nv_bfloat16*>(a.kcache);
  const __nv_bfloat16* vc = reinterpret_cast<const __nv_bfloat16*>(a.vcache);
  auto grow = [&](int slot) -> size_t {
    if constexpr (KIND == 1) return kv_row(a.page, seq, a.nkv, kvh, a.cap, slot);
    else return ((size_t)seq * a.nkv + kvh) * (size_t)a.cap + slot;
  };
  // keys k0 .. k1 - 1 of the staging order (region A: plain slots lo + k; region B: tree slot
  // ctx + k - nA)
  auto stage = [&](int k0, int k1) {
    constexpr int CH = D / 8;
    for (int i = threadIdx.x + k0 * CH; i < k1 * CH; i += blockDim.x) {
      const int k = i / CH, c = i % CH;
      const bool inA = k < nA;
      const int slot = inA ? lo + k : ctx + (k - nA);
      const bool ok = slot >= 0 && slot < a.cap;
      const size_t g = (ok ? grow(slot) : 0) * D + c * 8;
      const uint4 kv = ok ? *reinterpret_cast<const uint4*>(kc + g) : make_uint4(0, 0, 0, 0);
      const uint4 vv = ok ? *reinterpret_cast<const uint4*>(vc + g) : make_uint4(0, 0, 0, 0);
      __nv_bfloat16* dk = inA ? sAK + (size_t)k * LD : sBK + (size_t)(k - nA) * LD;
      __nv_bfloat16* dv = inA ? sAV + (size_t)k * LD : sBV + (size_t)(k - nA) * LD;
      *reinterpret_cast<uint4*>(dk + c * 8) = kv;
      *reinterpret_cast<uint4*>(dv + c * 8) = vv;
    }
  };
  if (pre) {
    stage(0, nA);
    PDL_ENTRY();
    stage(nA, nA + nB);
  } else {
    stage(0, nA);
  }
  __syncthreads();
  // per-warp scratch: the tail scores / probabilities and the key and value row pointers;
  // tail_cap is a multiple of 4, so every part starts on a 16-byte boundary
  const size_t wsz = (size_t)tail_cap * (4 + 16);
  float* wp = reinterpret_cast<float*>(wbase + (size_t)warp * wsz);
  const __nv_bfloat16** wk = reinterpret_cast<const __nv_bfloat16**>(wp + tail_cap);
  const __nv_bfloat16** wv = wk + tail_cap;
  const float sl2 = a.scale * 1.4426950408889634f;
  const int kg = lane >> 2, qt = lane & 3;
  for (int li = warp; li < n_items; li += blockDim.x / 32) {
    const int it = it0 + li;
    const int row = r0 + it / G, head = kvh * G + it % G;
    const int i = row - ra;
    const int P = s_P[i], pe = s_pe[i], body = s_body[i];
    const int nt = P + 1 - body;
    if (nt < 1 || nt > tail_cap) {             // a mask or slot the row layout does not allow
      if (lane == 0) latch_error(a.err, DEVERR_BOUNDS);
      continue;
    }
    // key and value rows of tail position body + j
    for (int j = lane; j < nt; j += 32) {
      const int p = body + j;
      const __nv_bfloat16 *kr, *vr;
      if (p < pe) {
        kr = sAK + (size_t)(p - lo) * LD;
        vr = sAV + (size_t)(p - lo) * LD;
      } else if (a.mode == 1) {
        // the (p - ctx)-th set bit of the row's ancestry mask
        int want = p - ctx, bit = 0;
        for (int w = 0; w < a.mask_words; ++w) {
          uint64_t m = a.mask[(size_t)row * a.mask_words + w];
          const int c = __popcll(m);
          if (want < c) {
            for (int q = 0; q < want; ++q) m &= m - 1;
            bit = w * 64 + __ffsll((long long)m) - 1;
            break;
          }
          want -= c;
        }
        if (bit < 0 || bit >= nB) {             // a mask bit past the tree
          latch_error(a.err, DEVERR_BOUNDS);
          bit = 0;
        }
        kr = sBK + (size_t)bit * LD;
        vr = sBV + (size_t)bit * LD;
      } else {
        const int t = pe - 1;                      // training-time test: own source chain
        const size_t gr = grow(ctx * (p - t) + t) * D;
        kr = kc + gr;
        vr = vc + gr;
      }
      wk[j] = kr;
      wv[j] = vr;
    }
    // this lane's quarter of the query vector
    float qv[DQ];
    {
      const __nv_bfloat16* qp = reinterpret_cast<const __nv_bfloat16*>(a.q) + ((size_t)row * a.nq + head) * D + qt * DQ;
#pragma unroll
      for (int c = 0; c < DQ; c += 8) {
        const uint4 raw = *reinterpret_cast<const uint4*>(qp + c);
        const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __bfloat1622float2(h2[e]);
          qv[c + 2 * e] = f.x;
          qv[c + 2 * e + 1] = f.y;
        }
      }
    }
    __syncwarp();
    // scores: key j by lanes 4 (j mod 8) .. +3, in passes of 8 keys
    for (int j0 = 0; j0 < nt; j0 += 8) {
      const int j = j0 + kg;
      float part = 0.f;
      if (j < nt) {
        const __nv_bfloat16* kr = wk[j] + qt * DQ;
        float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
        for (int c = 0; c < DQ; c += 8) {
          const uint4 raw = *reinterpret_cast<const uint4*>(kr + c);
          const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(h2[e]);
            acc0 = fmaf(qv[c + 2 * e], f.x, acc0);
            acc1 = fmaf(qv[c + 2 * e + 1], f.y, acc1);
          }
        }
        part = acc0 + acc1;
      }
      // (q0 + q1) + (q2 + q3): additions commute, so all four lanes hold the same value
      part += __shfl_xor_sync(0xffffffffu, part, 1);
      part += __shfl_xor_sync(0xffffffffu, part, 2);
      if (j < nt && qt == 0) wp[j] = part * sl2;
    }
    __syncwarp();
    float mt = -INFINITY;
    for (int j = lane; j < nt; j += 32) mt = fmaxf(mt, wp[j]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
    float lt = 0.f;
    for (int j = lane; j < nt; j += 32) {
      const float pj = exp2f(wp[j] - mt);
      wp[j] = pj;
      lt += pj;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lt += __shfl_xor_sync(0xffffffffu, lt, off);
    __syncwarp();
    float ot[DL];
#pragma unroll
    for (int u = 0; u < DL; ++u) ot[u] = 0.f;
    for (int j = 0; j < nt; ++j) {
      const float pj = wp[j];
      const __nv_bfloat16* vr = wv[j];
#pragma unroll
      for (int u = 0; u < DL; ++u) ot[u] = fmaf(pj, __bfloat162float(vr[lane + 32 * u]), ot[u]);
    }
    // the tail's partial goes right after the row's body splits
    const int sq = body > 0 ? (body + tps * MT_KEYS - 1) / (tps * MT_KEYS) : 0;
    const size_t q = ((size_t)sq * a.R + row) * a.nq + head;
#pragma unroll
    for (int u = 0; u < DL; ++u) a.part_o[q * D + lane + 32 * u] = ot[u];
    if (lane == 0) {
      a.part_ml[q * 2] = mt;
      a.part_ml[q * 2 + 1] = lt;
    }
    __syncwarp();
  }
}

// Body splits and tails: CTA (KV head, block of rows, z). z < splits: key split z of the
// block's bodies; z >= splits: tail chunk z - splits. Query vectors qv = (row - r0) * G + g.
// A body CTA writes the split's (m, l, o) of every query vector whose body reaches into it.
// KIND: 0 = contiguous cache, 1 = paged cache.
template <int D, int KIND, int NW>
__global__ void __launch_bounds__(NW * 32, NW == 4 ? 3 : 2)
    attn_split_k(AttnArgs a, int tps, int splits, int nB, int tail_cap) {
  constexpr int LD = D + 8;                      // padded smem row (bf16 elements)
  constexpr int QV = NW * 16;                    // query vectors per CTA
  constexpr int NT = NW * 32;
  extern __shared__ __align__(16) uint8_t attn_smem[];
  __nv_bfloat16* sK = reinterpret_cast<__nv_bfloat16*>(attn_smem);              // [2][64][LD]
  __nv_bfloat16* sV = sK + 2 * MT_KEYS * LD;                                    // [2][64][LD]
  __shared__ int s_body[QV];
  const int G = a.nq / a.nkv;
  const int RB = QV / G;
  const int nb = (a.rows_per_seq + RB - 1) / RB;
  const int kvh = blockIdx.x;
  const int sidx = blockIdx.y / nb, rb = blockIdx.y % nb;
  const int split = blockIdx.z;
  const int r0 = sidx * a.rows_per_seq + rb * RB;
  const int r1 = min(r0 + RB, min((sidx + 1) * a.rows_per_seq, a.R));
  if (r0 >= r1) return;
  if (split >= splits) {
    tail_chunk<D, KIND>(a, tps, r0, r1, kvh, split - splits, nB, tail_cap, attn_smem);
    return;
  }
  // Row metadata and context length were written before the preceding kernel started.
  const int seq = a.row_seq[r0];
  const int ctx = a.ctx_len[seq];
  // tree rows' bodies end at or before the context length: a split past it has nothing to do
  if (a.mode == 1 && split * tps * MT_KEYS >= ctx) return;
  for (int i = threadIdx.x; i < r1 - r0; i += blockDim.x) s_body[i] = row_span(a, r0 + i, ctx).body;
  __syncthreads();
  int bmax = 0;
  for (int i = 0; i < r1 - r0; ++i) bmax = max(bmax, s_body[i]);
  bmax = min(bmax, a.cap);
  const int t_begin = split * tps, t_end = min(t_begin + tps, (bmax + MT_KEYS - 1) / MT_KEYS);
  if (t_begin >= t_end) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const __nv_bfloat16* kc = reinterpret_cast<const __nv_bfloat16*>(a.kcache);
  const __nv_bfloat16* vc = reinterpret_cast<const __nv_bfloat16*>(a.vcache);

  // the two query vectors (rows of the mma fragment) this thread holds
  const int qv_a = warp * 16 + (lane >> 2), qv_b = qv_a + 8;
  const int row_a = r0 + qv_a / G, head_a = kvh * G + qv_a % G;
  const int row_b = r0 + qv_b / G, head_b = kvh * G + qv_b % G;
  const bool val_a = row_a < r1, val_b = row_b < r1;
  const int body_a = val_a ? s_body[row_a - r0] : 0, body_b = val_b ? s_body[row_b - r0] : 0;

  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;
  const float sl2 = a.scale * 1.4426950408889634f;

  // contiguous cache: one (sequence, head) run of rows; paged: rows through the block table
  const size_t head_row0 = KIND == 1 ? 0 : ((size_t)seq * a.nkv + kvh) * (size_t)a.cap;
  auto load_tile = [&](int t, int buf) {
    constexpr int CH = D / 8;   // 16-byte chunks per row
    for (int i = threadIdx.x; i < MT_KEYS * CH; i += NT) {
      const int kr = i / CH, c = i % CH;
      const int key = t * MT_KEYS + kr;
      const bool in = key < bmax;
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

  // Body keys sit below every slot the preceding kernel writes in tree mode (it writes the
  // tree rows' slots, from ctx on) and in one-row-per-sequence causal launches (it writes
  // the row's own slot, beyond its body): their first tile is requested before waiting.
  const bool early = a.mode == 1 || (a.mode == 0 && a.rows_per_seq == 1);
  if (early) load_tile(t_begin, 0);
  PDL_ENTRY();
  // Q fragments (bf16 pairs), zero for rows past the block
  uint32_t qf[D / 16][4];
  {
    const __nv_bfloat16* qp = reinterpret_cast<const __nv_bfloat16*>(a.q);
    const __nv_bfloat16* pa = qp + ((size_t)(val_a ? row_a : r0) * a.nq + head_a) * D;
    const __nv_bfloat16* pb = qp + ((size_t)(val_b ? row_b : r0) * a.nq + head_b) * D;
    const int c = (lane & 3) * 2;
#pragma unroll
    for (int kt = 0; kt < D / 16; ++kt) {
      qf[kt][0] = val_a ? *reinterpret_cast<const uint32_t*>(pa + kt * 16 + c) : 0u;
      qf[kt][1] = val_b ? *reinterpret_cast<const uint32_t*>(pb + kt * 16 + c) : 0u;
      qf[kt][2] = val_a ? *reinterpret_cast<const uint32_t*>(pa + kt * 16 + 8 + c) : 0u;
      qf[kt][3] = val_b ? *reinterpret_cast<const uint32_t*>(pb + kt * 16 + 8 + c) : 0u;
    }
  }
  if (!early) load_tile(t_begin, 0);
  const bool warp_live = warp * 16 < (r1 - r0) * G;
  for (int t = t_begin; t < t_end; ++t) {
    const int buf = (t - t_begin) & 1;
    if (t + 1 < t_end) { load_tile(t + 1, buf ^ 1); cp_async_wait<1>(); }
    else cp_async_wait<0>();
    __syncthreads();
    // a warp whose 16 query vectors are all past the block's rows only helps load the tiles
    if (!warp_live) { __syncthreads(); continue; }
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
    // keys past a query vector's body are its tail's or invisible: scaled to the exp2 domain
    // or -inf, then the running max
    float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int key = t * MT_KEYS + nt * 8 + (lane & 3) * 2 + e;
        s[nt][e] = key < body_a ? s[nt][e] * sl2 : -INFINITY;
        s[nt][2 + e] = key < body_b ? s[nt][2 + e] * sl2 : -INFINITY;
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
  const bool wr_a = val_a && t_begin * MT_KEYS < body_a, wr_b = val_b && t_begin * MT_KEYS < body_b;
  const size_t sa = ((size_t)split * a.R + row_a) * a.nq + head_a;
  const size_t sb = ((size_t)split * a.R + row_b) * a.nq + head_b;
#pragma unroll
  for (int i = 0; i < D / 8; ++i) {
    if (wr_a) *reinterpret_cast<float2*>(a.part_o + sa * D + i * 8 + c) = make_float2(o[i][0], o[i][1]);
    if (wr_b) *reinterpret_cast<float2*>(a.part_o + sb * D + i * 8 + c) = make_float2(o[i][2], o[i][3]);
  }
  if ((lane & 3) == 0) {
    if (wr_a) { a.part_ml[sa * 2] = m_a; a.part_ml[sa * 2 + 1] = l_a; }
    if (wr_b) { a.part_ml[sb * 2] = m_b; a.part_ml[sb * 2 + 1] = l_b; }
  }
}

// ---- body splits on the 5th-generation tensor cores (head dim 128) -------------------------------
// One CTA per (KV head, block of up to 128 query vectors, key split), 320 threads: warps 0-7
// are the softmax threads, two per query vector (TMEM lane = query vector; warp w takes lane
// quarter w % 4 and half w / 4 of the tile's keys and of O's columns), warp 8 issues the TMA
// loads, warp 9 the MMAs and owns the TMEM. Per 64-key tile t of the split:
//   S = Q K_t^T     tcgen05.mma, Q [128 x 128] and K_t [64 x 128] K-major in shared memory
//                   (128-byte swizzle), S [128 x 64] fp32 in TMEM;
//   softmax         each thread reads its half of its row of S, masks keys past its body,
//                   takes the row max with its partner (shared memory), updates its running
//                   max and its half's sum, and writes P = exp2(S - max) as a bf16 high part
//                   and a bf16 residual (~16 bits of P) to shared memory;
//   O += P V_t      two tcgen05.mma (high, residual) accumulate into O [128 x 128] fp32 in
//                   TMEM, V_t [64 keys x 128] read MN-major; before them the thread rescales
//                   its row of O when its max moved (a factor of exactly 1 is skipped).
// K_t+1 is loaded as soon as S_t is computed and V_t+1 as soon as O has taken V_t; S_t+1 is
// issued before P_t V_t, so the tensor cores compute it while the softmax of tile t ends.
// Every wait is bounded; a timeout latches an error and the CTA drains and exits.
constexpr int TC_SW = 2;                           // softmax threads per query vector
constexpr int TC_SOFT = 128 * TC_SW;               // softmax threads (warps 0 .. 4 TC_SW - 1)
constexpr int TC_THREADS = TC_SOFT + 64;           // + the TMA warp and the MMA warp
constexpr int TC_TAIL_ITEMS = 4 * (TC_THREADS / 32);   // tail items per CTA: four per warp
constexpr int TC_Q_BYTES = 2 * 128 * 128;          // [2 d-halves][128 rows][128 B]
constexpr int TC_KV_BYTES = 2 * 64 * 128;          // [2 d-halves][64 keys][128 B]
constexpr int TC_P_BYTES = 128 * 128;              // [128 rows][64 keys bf16]
constexpr int TC_SMEM = 1024 + TC_Q_BYTES + 2 * TC_KV_BYTES + 2 * TC_P_BYTES + 256;

// kind::f16 instruction descriptor: bf16 operands, fp32 accumulator, M = 128, N = n; A
// K-major; B K-major, or MN-major (transposed) when b_mn.
__device__ __forceinline__ constexpr uint32_t attn_idesc(int n, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (b_mn ? (1u << 16) : 0u) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(128 >> 4) << 24);
}

// MN-major operand with the 128-byte swizzle: rows of 64 MN-elements (128 bytes), one row
// per k; 8-row atoms 1024 bytes apart along k (stride byte offset), the next 64 MN-elements
// `mn_stride` bytes on (leading byte offset).
__device__ __forceinline__ uint64_t sdesc_sw128_mn(uint32_t saddr, uint32_t mn_stride) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFF) >> 4);
  d |= (uint64_t)((mn_stride >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* v) {
  tmem_st16(taddr, v);
  tmem_st16(taddr + 16, v + 16);
}

// A bounded wait taken by lane 0 for its warp: the warp's tcgen05.ld/st are collective
// (.sync.aligned), so every lane must take the same branch after a wait.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* err) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort_flag, err) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0;
}

// Whether every softmax thread's `ok` holds (a barrier of the TC_SOFT softmax threads with an
// AND reduction): the softmax warps leave the tile loop together, so their later barriers match.
__device__ __forceinline__ bool soft_all(bool ok) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)ok), "n"(TC_SOFT)
      : "memory");
  return r != 0;
}

template <int KIND>
__global__ void __launch_bounds__(TC_THREADS, 2)
    attn_tc_k(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, AttnArgs a,
              int tps, int splits, int nB, int tail_cap) {
  constexpr int D = 128;
  extern __shared__ __align__(16) uint8_t attn_smem[];
  const int G = a.nq / a.nkv;
  const int RB = 128 / G;
  const int nb = (a.rows_per_seq + RB - 1) / RB;
  const int kvh = blockIdx.x;
  const int sidx = blockIdx.y / nb, rb = blockIdx.y % nb;
  const int split = blockIdx.z;
  const int r0 = sidx * a.rows_per_seq + rb * RB;
  const int r1 = min(r0 + RB, min((sidx + 1) * a.rows_per_seq, a.R));
  if (r0 >= r1) return;
  if (split >= splits) {
    tail_chunk<D, KIND, TC_TAIL_ITEMS>(a, tps, r0, r1, kvh, split - splits, nB, tail_cap, attn_smem);
    return;
  }
  __shared__ int s_body[128];
  const int seq = a.row_seq[r0];
  const int ctx = a.ctx_len[seq];
  if (a.mode == 1 && split * tps * MT_KEYS >= ctx) return;
  for (int i = threadIdx.x; i < r1 - r0; i += blockDim.x) s_body[i] = row_span(a, r0 + i, ctx).body;
  __syncthreads();
  int bmax = 0;
  for (int i = 0; i < r1 - r0; ++i) bmax = max(bmax, s_body[i]);
  bmax = min(bmax, a.cap);
  const int t_begin = split * tps, t_end = min(t_begin + tps, (bmax + MT_KEYS - 1) / MT_KEYS);
  if (t_begin >= t_end) return;

  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(attn_smem) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = sm;
  uint8_t* sK = sQ + TC_Q_BYTES;
  uint8_t* sV = sK + TC_KV_BYTES;
  uint8_t* sP = sV + TC_KV_BYTES;                       // [hi, lo]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sP + 2 * TC_P_BYTES);
  uint64_t* k_full = bars + 0;
  uint64_t* k_empty = bars + 1;
  uint64_t* v_full = bars + 2;
  uint64_t* v_empty = bars + 3;
  uint64_t* s_full = bars + 4;
  uint64_t* s_empty = bars + 5;
  uint64_t* p_full = bars + 6;
  uint64_t* o_done = bars + 7;    // P_t V_t complete (O updated, P and V_t free)
  uint64_t* q_ready = bars + 8;
  uint64_t* drain = bars + 9;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 10);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt = t_end - t_begin;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(k_full), 1);
    mbar_init(smem_u32(k_empty), 1);
    mbar_init(smem_u32(v_full), 1);
    mbar_init(smem_u32(v_empty), 1);
    mbar_init(smem_u32(s_full), 1);
    mbar_init(smem_u32(s_empty), TC_SOFT);
    mbar_init(smem_u32(p_full), TC_SOFT);
    mbar_init(smem_u32(o_done), 1);
    mbar_init(smem_u32(q_ready), TC_SOFT);
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  constexpr int W_TMA = TC_SOFT / 32, W_MMA = W_TMA + 1;
  if (warp == W_MMA) tmem_alloc(smem_u32(tmem_slot), 256);   // S: columns 0-63, O: 128-255
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const size_t head_row0 = KIND == 1 ? 0 : ((size_t)seq * a.nkv + kvh) * (size_t)a.cap;

  if (warp == W_TMA) {
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      // a tile's rows: one 64-row box per d-half (contiguous cache) or one 16-row box per
      // cache block (paged); boxes wholly past the keys in use are not loaded
      auto load_tile = [&](const CUtensorMap* map, uint8_t* dst, int t, uint32_t bar) {
        if constexpr (KIND == 0) {
          mbar_expect_tx(bar, TC_KV_BYTES);
          const int row = (int)(head_row0 + (size_t)t * MT_KEYS);
          tma_load_2d(smem_u32(dst), map, 0, row, bar, pol);
          tma_load_2d(smem_u32(dst + TC_KV_BYTES / 2), map, 64, row, bar, pol);
        } else {
          const int box = min(1 << a.page.bs_log2, MT_KEYS);   // slots of a block are consecutive rows
          const int nbox = MT_KEYS / box;
          int live = 0;
          for (int i = 0; i < nbox; ++i) live += (t * MT_KEYS + i * box < bmax);
          mbar_expect_tx(bar, (uint32_t)live * box * 256);
          for (int i = 0; i < nbox; ++i) {
            const int slot = t * MT_KEYS + i * box;
            if (slot >= bmax) continue;
            const int row = (int)kv_row(a.page, seq, a.nkv, kvh, a.cap, slot);
            tma_load_2d(smem_u32(dst + i * box * 128), map, 0, row, bar, pol);
            tma_load_2d(smem_u32(dst + TC_KV_BYTES / 2 + i * box * 128), map, 64, row, bar, pol);
          }
        }
      };
      // K and V of the first tile sit below every slot the preceding kernel writes only in
      // tree mode; wait for it before the first load otherwise
      if (a.mode != 1) pdl_wait();
      load_tile(&tmK, sK, t_begin, smem_u32(k_full));
      load_tile(&tmV, sV, t_begin, smem_u32(v_full));
      int nk = 1, nv = 1;   // tiles issued
      for (int i = 1; i < nt; ++i) {
        const uint32_t ph = (uint32_t)((i - 1) & 1);
        if (!mbar_wait(smem_u32(k_empty), ph, abort_flag, a.err)) break;
        load_tile(&tmK, sK, t_begin + i, smem_u32(k_full));
        ++nk;
        if (!mbar_wait(smem_u32(v_empty), ph, abort_flag, a.err)) break;
        load_tile(&tmV, sV, t_begin + i, smem_u32(v_full));
        ++nv;
      }
      if (*abort_flag) {   // let the copies in flight land before the CTA leaves
        mbar_wait(smem_u32(k_full), (uint32_t)((nk - 1) & 1), abort_flag, a.err, false);
        mbar_wait(smem_u32(v_full), (uint32_t)((nv - 1) & 1), abort_flag, a.err, false);
      }
    }
  } else if (warp == W_MMA) {
    if (lane == 0) {
      constexpr uint32_t IS = attn_idesc(64, false), IO = attn_idesc(128, true);
      const uint32_t tS = tmem, tO = tmem + 128;
      bool ok = mbar_wait(smem_u32(q_ready), 0, abort_flag, a.err);
      auto issue_s = [&](int i) -> bool {
        if (!mbar_wait(smem_u32(k_full), (uint32_t)(i & 1), abort_flag, a.err)) return false;
        if (i > 0 && !mbar_wait(smem_u32(s_empty), (uint32_t)((i - 1) & 1), abort_flag, a.err)) return false;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t da = sdesc_sw128(smem_u32(sQ + (k >> 2) * (TC_Q_BYTES / 2) + (k & 3) * 32));
          const uint64_t db = sdesc_sw128(smem_u32(sK + (k >> 2) * (TC_KV_BYTES / 2) + (k & 3) * 32));
          tc_mma_bf16(tS, da, db, IS, k ? 1u : 0u);
        }
        tc_commit(smem_u32(s_full));
        tc_commit(smem_u32(k_empty));
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int i = 0; ok && i < nt; ++i) {
        if (i + 1 < nt && !issue_s(i + 1)) { ok = false; break; }
        if (!mbar_wait(smem_u32(p_full), (uint32_t)(i & 1), abort_flag, a.err) ||
            !mbar_wait(smem_u32(v_full), (uint32_t)(i & 1), abort_flag, a.err)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int part = 0; part < 2; ++part)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint64_t da = sdesc_sw128(smem_u32(sP + part * TC_P_BYTES + j * 32));
            const uint64_t db = sdesc_sw128_mn(smem_u32(sV + j * 2048), TC_KV_BYTES / 2);
            tc_mma_bf16(tO, da, db, IO, (i > 0 || part || j) ? 1u : 0u);
          }
        tc_commit(smem_u32(o_done));
        tc_commit(smem_u32(v_empty));
      }
      if (!ok) {
        tc_commit(smem_u32(drain));
        mbar_wait(smem_u32(drain), 0, abort_flag, a.err, false);
      }
    }
  } else {
    // softmax threads: query vector qv (TMEM lane), half h of the keys and of O's columns
    constexpr int SC = 64 / TC_SW, OC = 128 / TC_SW;   // S and O columns per thread
    __shared__ float x_max[2][TC_SW][128];             // partner exchange, by tile parity
    __shared__ float x_l[TC_SW][128];
    const int qv = threadIdx.x & 127, h = threadIdx.x >> 7;
    const int row = r0 + qv / G, head = kvh * G + qv % G;
    const bool valid = row < r1;
    const int body = valid ? s_body[row - r0] : 0;
    PDL_ENTRY();
    {
      // Q row -> shared memory, 128-byte swizzle (16-byte chunk c of row r at c ^ (r & 7));
      // this thread's half of the head dimension
      const uint4* qp = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(a.q) +
                                                       ((size_t)(valid ? row : r0) * a.nq + head) * D);
#pragma unroll
      for (int k = 0; k < 16 / TC_SW; ++k) {
        const int c = h * (16 / TC_SW) + k;
        const uint4 x = valid ? qp[c] : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(sQ + (c >> 3) * (TC_Q_BYTES / 2) + qv * 128 + (((c & 7) ^ (qv & 7)) << 4)) = x;
      }
      fence_proxy_async_all();
      mbar_arrive(smem_u32(q_ready));
    }
    const uint32_t lane_off = (uint32_t)(((warp & 3) * 32) << 16);
    const uint32_t tS = tmem + lane_off + h * SC, tO = tmem + 128 + lane_off + h * OC;
    const float sl2 = a.scale * 1.4426950408889634f;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int i = 0; i < nt; ++i) {
      const int t = t_begin + i;
      const bool got = warp_wait(smem_u32(s_full), (uint32_t)(i & 1), abort_flag, a.err);
      float s[SC];
      if (got) {
        tc_fence_after();
        tmem_ld32(tS, s);
        tc_fence_before();
        mbar_arrive(smem_u32(s_empty));
      } else {
#pragma unroll
        for (int j = 0; j < SC; ++j) s[j] = 0.f;
      }
      // keys past this query vector's body belong to its tail or are invisible
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < SC; ++j) {
        s[j] = t * MT_KEYS + h * SC + j < body ? s[j] * sl2 : -INFINITY;
        mx = fmaxf(mx, s[j]);
      }
      // the row max over both halves (the partner holds the other half); the same barrier
      // tells every softmax thread whether all waits held
      x_max[i & 1][h][qv] = mx;
      if (!soft_all(got)) { ok = false; break; }
      mx = fmaxf(x_max[i & 1][0][qv], x_max[i & 1][1][qv]);
      const float mn = fmaxf(m, mx);
      const float base = mn == -INFINITY ? 0.f : mn;
      const float corr = exp2f(m - base);
      m = mn;
      float ps = 0.f;
#pragma unroll
      for (int j = 0; j < SC; ++j) {
        s[j] = exp2f(s[j] - base);
        ps += s[j];
      }
      l = l * corr + ps;
      // P_(t-1) V_(t-1) must be complete before O is rescaled and P is overwritten
      if (i > 0) {
        if (!soft_all(warp_wait(smem_u32(o_done), (uint32_t)((i - 1) & 1), abort_flag, a.err))) {
          ok = false;
          break;
        }
        tc_fence_after();
        // warp-uniform: a lane whose factor is exactly 1 multiplies by 1
        if (__any_sync(0xffffffffu, corr != 1.f)) {
#pragma unroll
          for (int c0 = 0; c0 < OC; c0 += 32) {
            float o[32];
            tmem_ld32(tO + c0, o);
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] *= corr;
            tmem_st32(tO + c0, o);
          }
          tmem_wait_st();
        }
      }
      // the last tile's keys past the block's bodies: V rows zeroed (P is zero there, and a
      // stale slot must not contribute 0 * NaN)
      if (t * MT_KEYS + MT_KEYS > bmax) {
        if (!soft_all(warp_wait(smem_u32(v_full), (uint32_t)(i & 1), abort_flag, a.err))) {
          ok = false;
          break;
        }
        const int k0 = bmax - t * MT_KEYS;
        for (int idx = threadIdx.x; idx < (MT_KEYS - k0) * 16; idx += TC_SOFT) {
          const int kr = k0 + idx / 16, c = idx % 16;
          *reinterpret_cast<uint4*>(sV + (c >> 3) * (TC_KV_BYTES / 2) + kr * 128 + ((c & 7) << 4)) =
              make_uint4(0, 0, 0, 0);
        }
      }
      // P (high part, then residual) -> shared memory, same swizzle as Q: this thread's keys
#pragma unroll
      for (int c = 0; c < SC / 8; ++c) {
        uint32_t hp[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) split_bf16(s[c * 8 + 2 * e], s[c * 8 + 2 * e + 1], hp[e], lo[e]);
        const int cc = h * (SC / 8) + c;
        const int off = qv * 128 + ((cc ^ (qv & 7)) << 4);
        *reinterpret_cast<uint4*>(sP + off) = make_uint4(hp[0], hp[1], hp[2], hp[3]);
        *reinterpret_cast<uint4*>(sP + TC_P_BYTES + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
      fence_proxy_async_all();
      tc_fence_before();
      mbar_arrive(smem_u32(p_full));
    }
    // the row's sum: the halves' running sums added in a fixed order
    x_l[h][qv] = l;
    named_bar_sync(1, TC_SOFT);
    l = x_l[0][qv] + x_l[1][qv];
    if (ok && warp_wait(smem_u32(o_done), (uint32_t)((nt - 1) & 1), abort_flag, a.err)) {
      tc_fence_after();
      const bool wr = valid && t_begin * MT_KEYS < body;
      const size_t q = ((size_t)split * a.R + row) * a.nq + head;
#pragma unroll
      for (int c0 = 0; c0 < OC; c0 += 32) {
        float o[32];
        tmem_ld32(tO + c0, o);
        if (wr) {
#pragma unroll
          for (int j = 0; j < 32; j += 4)
            *reinterpret_cast<float4*>(a.part_o + q * D + h * OC + c0 + j) =
                make_float4(o[j], o[j + 1], o[j + 2], o[j + 3]);
        }
      }
      if (wr && h == 0) {
        a.part_ml[q * 2] = m;
        a.part_ml[q * 2 + 1] = l;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == W_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// Merge: one warp per (row, query head). Lane s holds partial s (the body splits of the
// row's position, then its tail); the weighted sums run in partial order.
template <int D>
__global__ void attn_merge_k(AttnArgs a, int tps) {
  constexpr int DL = D / 32;
  const int qi = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  // the row's span reads row metadata only, which the preceding (attention) kernel does not
  // write: it is computed before the wait
  const int row = min(qi, a.R * a.nq - 1) / a.nq;
  const int body = row_span(a, row, a.ctx_len[a.row_seq[row]]).body;
  PDL_ENTRY();
  if (qi >= a.R * a.nq) return;
  const int S = (body > 0 ? (body + tps * MT_KEYS - 1) / (tps * MT_KEYS) : 0) + 1;   // <= 32
  const size_t stride = (size_t)a.R * a.nq;
  float ms = -INFINITY, ls = 0.f;
  if (lane < S) {
    ms = a.part_ml[((size_t)lane * stride + qi) * 2];
    ls = a.part_ml[((size_t)lane * stride + qi) * 2 + 1];
  }
  float M = ms;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  const float ws = lane < S ? exp2f(ms - M) : 0.f;
  const float lw = ls * ws;
  float L = 0.f, acc[DL];
#pragma unroll
  for (int u = 0; u < DL; ++u) acc[u] = 0.f;
  for (int s0 = 0; s0 < S; s0 += 8) {
    float x[8][DL];
#pragma unroll
    for (int k = 0; k < 8; ++k)
#pragma unroll
      for (int u = 0; u < DL; ++u)
        x[k][u] = s0 + k < S ? a.part_o[((size_t)(s0 + k) * stride + qi) * D + lane + 32 * u] : 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float w = __shfl_sync(0xffffffffu, ws, (s0 + k) & 31);
      const float l = __shfl_sync(0xffffffffu, lw, (s0 + k) & 31);
      if (s0 + k < S) {
        L += l;
#pragma unroll
        for (int u = 0; u < DL; ++u) acc[u] = fmaf(x[k][u], w, acc[u]);
      }
    }
  }
  __nv_bfloat16* op = reinterpret_cast<__nv_bfloat16*>(a.out) + (size_t)qi * D;
#pragma unroll
  for (int u = 0; u < DL; ++u) op[lane + 32 * u] = __float2bfloat16_rn(L > 0.f ? acc[u] / L : 0.f);
}

size_t attention_scratch_floats(int rows, int nq, int d) { return (size_t)(MAX_SPLITS + 1) * rows * nq * (d + 2); }

// Key splits of a cache of `cap` slots serving up to `batch` sequences: three 64-key tiles
// per split for one to seven sequences (more splits put the merge and the CTA count on the
// critical path, fewer lengthen each CTA: measured on the 8B batch-1 verify pass), eight
// from eight sequences on, where the sequences and heads alone fill the GPU and shorter
// splits only add partials; at most MAX_SPLITS.
int attention_max_splits(int cap, int batch) {
  const int tiles = (cap + MT_KEYS - 1) / MT_KEYS;
  const int per = batch >= 8 ? 8 : 3;
  return std::max(1, std::min(MAX_SPLITS, (tiles + per - 1) / per));
}

template <int D, int NW>
static int launch_bf16(cudaStream_t st, const AttnArgs& a) {
  const int G = a.nq / a.nkv;
  const int RB = NW * 16 / G;
  const int nseq = (a.R + a.rows_per_seq - 1) / a.rows_per_seq;
  const int nb = (a.rows_per_seq + RB - 1) / RB;
  if (!a.part_o || !a.part_ml) return -1;
  // fixed key splits: a function of the capacity and the caller's constant only; partials
  // hold the splits and one tail slot per row
  const int max_tiles = std::max(1, (a.cap + MT_KEYS - 1) / MT_KEYS);
  const long long fit = (long long)(a.part_floats / ((size_t)a.R * a.nq * D)) - 1;
  if (fit < 1) return -1;
  const int S = (int)std::min<long long>(std::min(MAX_SPLITS, std::max(1, a.max_splits)), fit);
  const int tps = (max_tiles + S - 1) / S;
  const int splits = (max_tiles + tps - 1) / tps;
  const int chunks = (RB * G + TAIL_ITEMS - 1) / TAIL_ITEMS;
  const int nB = a.mode == 1 ? a.tree_T : 0;
  const int tail_cap = (std::max(TAIL_MIN, a.mode == 1 ? a.tree_T : 0) + 3) & ~3;   // a multiple of 4
  const size_t body_smem = (size_t)4 * MT_KEYS * (D + 8) * sizeof(__nv_bfloat16);
  const size_t tail_smem = (size_t)2 * (TAIL_MIN + TAIL_ITEMS + nB) * (D + 8) * sizeof(__nv_bfloat16) +
                           (size_t)NW * tail_cap * (4 + 16);
  const size_t smem = std::max(body_smem, tail_smem);
  const bool paged = a.page.table != nullptr;
  const void* fn = paged ? reinterpret_cast<const void*>(attn_split_k<D, 1, NW>)
                         : reinterpret_cast<const void*>(attn_split_k<D, 0, NW>);
  if (raise_smem_limit(fn, (int)smem) != cudaSuccess) return -4;
  const dim3 grid(a.nkv, nseq * nb, splits + chunks);
  if (paged) launch_k(attn_split_k<D, 1, NW>, grid, NW * 32, smem, st, a, tps, splits, nB, tail_cap);
  else launch_k(attn_split_k<D, 0, NW>, grid, NW * 32, smem, st, a, tps, splits, nB, tail_cap);
  launch_k(attn_merge_k<D>, (a.R * a.nq + 3) / 4, 128, 0, st, a, tps);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

// Which bodies run head dim 128: mma.sync by default, tcgen05 with EAGLE_ATTN_TC=1 (the two
// sum in different orders, so the setting holds for the whole process and every launch over a
// cache agrees). The tcgen05 bodies win on tree rows alone (batch 64 x 1100 keys x 17 rows:
// 239 against 275 us; batch 8 x 2048 keys: 45 against 53 us) but lose on the one-row steps of
// plain decoding, which must use the same bodies (a 128-row MMA tile holding 4 query vectors:
// batch-64 plain step 10.8 against 6.9 ms), and on the 61-row batch-1 tree (35 against 23 us);
// the batch-64 cycle as a whole: 34.7 against 34.1 ms.
static bool tc_bodies(const AttnArgs&) {
  static const bool on = getenv("EAGLE_ATTN_TC") && strcmp(getenv("EAGLE_ATTN_TC"), "1") == 0;
  return on;
}

// Head dim 128 with the cache's row count known: bodies on tcgen05 (attn_tc_k).
static int launch_tc(cudaStream_t st, const AttnArgs& a) {
  constexpr int D = 128;
  const int G = a.nq / a.nkv;
  const int RB = 128 / G;
  const int nseq = (a.R + a.rows_per_seq - 1) / a.rows_per_seq;
  const int nb = (a.rows_per_seq + RB - 1) / RB;
  if (!a.part_o || !a.part_ml) return -1;
  const int max_tiles = std::max(1, (a.cap + MT_KEYS - 1) / MT_KEYS);
  const long long fit = (long long)(a.part_floats / ((size_t)a.R * a.nq * D)) - 1;
  if (fit < 1) return -1;
  const int S = (int)std::min<long long>(std::min(MAX_SPLITS, std::max(1, a.max_splits)), fit);
  const int tps = (max_tiles + S - 1) / S;
  const int splits = (max_tiles + tps - 1) / tps;
  const int chunks = (RB * G + TC_TAIL_ITEMS - 1) / TC_TAIL_ITEMS;
  const int nB = a.mode == 1 ? a.tree_T : 0;
  const int tail_cap = (std::max(TAIL_MIN, a.mode == 1 ? a.tree_T : 0) + 3) & ~3;
  const size_t tail_smem = (size_t)2 * (TAIL_MIN + TC_TAIL_ITEMS + nB) * (D + 8) * sizeof(__nv_bfloat16) +
                           (size_t)(TC_THREADS / 32) * tail_cap * (4 + 16);
  const size_t smem = std::max((size_t)TC_SMEM, tail_smem);
  const bool paged = a.page.table != nullptr;
  const int box = paged ? std::min(1 << a.page.bs_log2, MT_KEYS) : MT_KEYS;
  CUtensorMap mk, mv;
  if (!make_tmap_bf16(&mk, a.kcache, a.kv_rows, D, box) || !make_tmap_bf16(&mv, a.vcache, a.kv_rows, D, box))
    return -4;
  const void* fn = paged ? reinterpret_cast<const void*>(attn_tc_k<1>) : reinterpret_cast<const void*>(attn_tc_k<0>);
  if (raise_smem_limit(fn, (int)smem) != cudaSuccess) return -4;
  const dim3 grid(a.nkv, nseq * nb, splits + chunks);
  if (paged) launch_k(attn_tc_k<1>, grid, TC_THREADS, smem, st, mk, mv, a, tps, splits, nB, tail_cap);
  else launch_k(attn_tc_k<0>, grid, TC_THREADS, smem, st, mk, mv, a, tps, splits, nB, tail_cap);
  launch_k(attn_merge_k<D>, (a.R * a.nq + 3) / 4, 128, 0, st, a, tps);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

// CTA size: 4 warps (64 query vectors), or 6 (96) when that puts all of a sequence's rows
// in one block that 4 warps would split in two (each block streams the sequence's keys;
// with more blocks, more and smaller CTAs measured faster). A query vector's arithmetic
// does not depend on the block it sits in: keys past its body are masked to exact zeros,
// so the choice is one of speed only.
template <int D>
static int launch_bf16_nw(cudaStream_t st, const AttnArgs& a, int G) {
  const int qv = a.rows_per_seq * G;
  const bool six = 96 % G == 0 && qv > 64 && qv <= 96;
  return six ? launch_bf16<D, 6>(st, a) : launch_bf16<D, 4>(st, a);
}

int attention_bf16_mma(cudaStream_t st, const AttnArgs& a) {
  const int G = a.nq / a.nkv;
  if (G < 1 || G > 64 || 64 % G) return -1;
  if (a.mode == 1 && (a.mask_words > 4 || a.tree_T > 256 || a.tree_T < 1)) return -1;
  if (a.mode == 2 && a.page.table) return -1;   // the training-time test runs on the contiguous drafter cache
  switch (a.d) {
    case 32: return launch_bf16_nw<32>(st, a, G);
    case 64: return launch_bf16_nw<64>(st, a, G);
    case 128: return a.kv_rows > 0 && 128 % G == 0 && tc_bodies(a) ? launch_tc(st, a) : launch_bf16_nw<128>(st, a, G);
  }
  return -1;
}

}  // namespace eagle
