// Row-wise fused ops of the Llama-style layer: embedding gather, RMSNorm, rotary
// embedding with the KV-cache write, SwiGLU, the drafter's [emb; feature] input, and
// plain row conversions / gathers. All are memory-bound and use coalesced row loops.
#include "common.cuh"
#include "kernels.h"
#include <type_traits>

namespace eagle {

template <typename T>
__global__ void embed_k(const T* E, int V, int H, const int* tok, float* x, int* err) {
  PDL_ENTRY();
  const int r = blockIdx.x;
  int t = tok[r];
  if (t < 0 || t >= V) {
    if (threadIdx.x == 0) latch_error(err, DEVERR_BOUNDS);
    t = 0;
  }
  const T* e = E + (size_t)t * H;
  float* o = x + (size_t)r * H;
  for (int base = 0; base < H; base += 4 * blockDim.x) {
    float v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i = base + k * blockDim.x + threadIdx.x;
      v[k] = i < H ? Elem<T>::to_f(e[i]) : 0.f;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i = base + k * blockDim.x + threadIdx.x;
      if (i < H) o[i] = v[k];
    }
  }
}

int embed_rows(cudaStream_t st, int dtype, const void* E, int V, int H, const int* tok, int R, float* x,
               int* err) {
  if (R <= 0) return 0;
  if (dtype == DT_F32) launch_k(embed_k<float>, R, 256, 0, st, (const float*)E, V, H, tok, x, err);
  else launch_k(embed_k<__nv_bfloat16>, R, 256, 0, st, (const __nv_bfloat16*)E, V, H, tok, x, err);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

// out = x / sqrt(mean(x^2) + eps) * g. One block per row; each thread keeps up to
// RN_PER_THREAD elements of the row in registers, so the row is read once. Fixed
// reduction order (per-thread sums, then a fixed warp/block tree).
constexpr int RN_THREADS = 256;
constexpr int RN_PER_THREAD = 24;   // rows up to 6144 elements stay in registers

// This thread's gains of a row of H (constants: they may be read before the dependency wait).
template <typename TG>
__device__ __forceinline__ void rms_gains(const TG* g, int H, float* gv) {
#pragma unroll
  for (int j = 0; j < RN_PER_THREAD; ++j) {
    const int i = threadIdx.x + j * RN_THREADS;
    gv[j] = i < H ? Elem<TG>::to_f(g[i]) : 0.f;
  }
}

// One row by RN_THREADS threads, with this thread's gains already loaded (shared by
// rmsnorm_k and the fused drafter-input kernel, so both give the same bits).
template <typename TX, typename TG, typename TO>
__device__ __forceinline__ void rms_row(const TX* xr, const TG* g, const float* gv, int H, float eps, TO* o) {
  float v[RN_PER_THREAD];
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < RN_PER_THREAD; ++j) {
    const int i = threadIdx.x + j * RN_THREADS;
    v[j] = i < H ? Elem<TX>::to_f(xr[i]) : 0.f;
  }
#pragma unroll
  for (int j = 0; j < RN_PER_THREAD; ++j) s = fmaf(v[j], v[j], s);
  for (int i = threadIdx.x + RN_PER_THREAD * RN_THREADS; i < H; i += RN_THREADS) {
    const float t = Elem<TX>::to_f(xr[i]);
    s = fmaf(t, t, s);
  }
  __shared__ float red[RN_THREADS / 32];
  s = warp_sum(s);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < RN_THREADS / 32; ++w) tot += red[w];
  const float rs = rsqrtf(tot / (float)H + eps);
#pragma unroll
  for (int j = 0; j < RN_PER_THREAD; ++j) {
    const int i = threadIdx.x + j * RN_THREADS;
    if (i < H) o[i] = Elem<TO>::from_f(v[j] * rs * gv[j]);
  }
  for (int i = threadIdx.x + RN_PER_THREAD * RN_THREADS; i < H; i += RN_THREADS)
    o[i] = Elem<TO>::from_f(Elem<TX>::to_f(xr[i]) * rs * Elem<TG>::to_f(g[i]));
}

template <typename TX, typename TG, typename TO>
__global__ void __launch_bounds__(RN_THREADS) rmsnorm_k(const TX* x, int ldx, const TG* g, int H, float eps, TO* out,
                                                        int ldo) {
  float gv[RN_PER_THREAD];
  rms_gains(g, H, gv);   // the gains before the wait, the row (the preceding kernel's output) after
  PDL_ENTRY();
  const int r = blockIdx.x;
  rms_row<TX, TG, TO>(x + (size_t)r * ldx, g, gv, H, eps, out + (size_t)r * ldo);
}

// EAGLE-3 drafter input of one row per block, in one pass (the bits of gather + widen +
// RMSNorm + embedding gather + RMSNorm): g = feature row feat_row[r] (row r when null) -> gbuf
// row r (when it is another buffer) and the fp32 residual x row r; ain row r =
// [RMSNorm(g) * norm_g ; RMSNorm(emb(tok)) * norm_e]; ebuf row r = emb(tok).
__global__ void __launch_bounds__(RN_THREADS)
    eagle3_input_k(const __nv_bfloat16* feat, const int* feat_row, const __nv_bfloat16* E, int V, const int* tok,
                   int H, const __nv_bfloat16* ng, const __nv_bfloat16* ne, float eps, __nv_bfloat16* gbuf, float* x,
                   __nv_bfloat16* ebuf, __nv_bfloat16* ain, int* err) {
  float gv[RN_PER_THREAD];
  rms_gains(ng, H, gv);
  PDL_ENTRY();
  const int r = blockIdx.x;
  const __nv_bfloat16* g = feat + (size_t)(feat_row ? feat_row[r] : r) * H;
  __nv_bfloat16* gr = gbuf + (size_t)r * H;
  float* xr = x + (size_t)r * H;
  for (int i = threadIdx.x; i < H; i += RN_THREADS) {
    const __nv_bfloat16 v = g[i];
    if (gr != g) gr[i] = v;
    xr[i] = __bfloat162float(v);
  }
  __nv_bfloat16* ar = ain + (size_t)r * 2 * H;
  rms_row<__nv_bfloat16, __nv_bfloat16, __nv_bfloat16>(g, ng, gv, H, eps, ar);
  __syncthreads();   // the reduction scratch is reused below
  int t = tok[r];
  if (t < 0 || t >= V) {
    if (threadIdx.x == 0) latch_error(err, DEVERR_BOUNDS);
    t = 0;
  }
  const __nv_bfloat16* e = E + (size_t)t * H;
  __nv_bfloat16* er = ebuf + (size_t)r * H;
  for (int i = threadIdx.x; i < H; i += RN_THREADS) er[i] = e[i];
  rms_gains(ne, H, gv);
  rms_row<__nv_bfloat16, __nv_bfloat16, __nv_bfloat16>(e, ne, gv, H, eps, ar + H);
}

int eagle3_input_rows(cudaStream_t st, const void* feat, const int* feat_row, const void* E, int V, const int* tok,
                      int H, const void* norm_g, const void* norm_e, float eps, void* gbuf, float* x, void* ebuf,
                      void* ain, int R, int* err) {
  if (R <= 0) return 0;
  launch_k(eagle3_input_k, R, RN_THREADS, 0, st, (const __nv_bfloat16*)feat, feat_row, (const __nv_bfloat16*)E, V,
           tok, H, (const __nv_bfloat16*)norm_g, (const __nv_bfloat16*)norm_e, eps, (__nv_bfloat16*)gbuf, x,
           (__nv_bfloat16*)ebuf, (__nv_bfloat16*)ain, err);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

int rmsnorm_rows(cudaStream_t st, int dtype_in, const void* x, int ldx, const void* g, int H, float eps,
                 int R, int dtype_out, void* out, int ldo) {
  if (R <= 0) return 0;
  // gains are stored in the model's storage type, which equals dtype_out
  if (dtype_out == DT_F32) {
    if (dtype_in != DT_F32) return -1;
    launch_k(rmsnorm_k<float, float, float>, R, RN_THREADS, 0, st, (const float*)x, ldx, (const float*)g, H, eps, (float*)out, ldo);
  } else if (dtype_in == DT_F32) {
    launch_k(rmsnorm_k<float, __nv_bfloat16, __nv_bfloat16>, R, RN_THREADS, 0, st, 
        (const float*)x, ldx, (const __nv_bfloat16*)g, H, eps, (__nv_bfloat16*)out, ldo);
  } else {
    launch_k(rmsnorm_k<__nv_bfloat16, __nv_bfloat16, __nv_bfloat16>, R, RN_THREADS, 0, st, 
        (const __nv_bfloat16*)x, ldx, (const __nv_bfloat16*)g, H, eps, (__nv_bfloat16*)out, ldo);
  }
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

// Rotate-half RoPE on q and k (angle table precomputed on the host in double precision);
// q written to q_out, k and v into the cache at the row's slot. One block per row and group
// of RS_HEADS heads of the fused [q | k | v] projection output; a thread takes RS_ITEMS
// (head, rotation pair) items, loading all of them before it stores.
constexpr int RS_HEADS = 8, RS_THREADS = 128, RS_ITEMS = 4;

template <typename T>
__global__ void rope_store_k(const float* qkv, int nq, int nkv, int d, const int* row_pos, const int* row_slot,
                             const int* row_seq, const float* rc, const float* rsn, T* q_out, T* kc, T* vc, int cap,
                             int* err, int slot_limit, KvPage page) {
  const int r = blockIdx.x, h0 = blockIdx.y * RS_HEADS;
  const int H = nq + 2 * nkv, half = d / 2;
  // The row's slot, position, block-table entry and angle table rows are written before the
  // preceding kernel (the projection): they are read before the wait, the projection's
  // output after it.
  const int slot = row_slot[r];
  // a paged cache must hold a block for the slot (assigned before the step that writes it)
  const bool slot_ok = slot >= 0 && slot < cap && slot < slot_limit &&
                       (!page.table || page.table[(size_t)row_seq[r] * page.tab_w + (slot >> page.bs_log2)] >= 0);
  const int seq = row_seq[r], pos = row_pos[r];
  const float* src = qkv + (size_t)r * H * d;
  const int n = min(RS_HEADS, H - h0) * half;   // (head, pair) items of this block
  float cs0[RS_ITEMS], sn0[RS_ITEMS];           // the first round's angles
#pragma unroll
  for (int k = 0; k < RS_ITEMS; ++k) {
    const int it = k * RS_THREADS + threadIdx.x;
    const int hl = it / half, i = it - hl * half, h = h0 + hl;
    cs0[k] = sn0[k] = 0.f;
    if (it < n && h < nq + nkv) {
      cs0[k] = rc[(size_t)pos * half + i];
      sn0[k] = rsn[(size_t)pos * half + i];
    }
  }
  PDL_ENTRY();
  if (!slot_ok && blockIdx.y == 0 && threadIdx.x == 0) latch_error(err, DEVERR_CAPACITY);
  for (int base = 0; base < n; base += RS_ITEMS * RS_THREADS) {
    // all loads of the thread's items first, then the rotations and stores
    float xa[RS_ITEMS], xb[RS_ITEMS], cs[RS_ITEMS], sn[RS_ITEMS];
#pragma unroll
    for (int k = 0; k < RS_ITEMS; ++k) {
      const int it = base + k * RS_THREADS + threadIdx.x;
      const int hl = it / half, i = it - hl * half, h = h0 + hl;
      xa[k] = xb[k] = 0.f;
      cs[k] = base == 0 ? cs0[k] : 0.f;
      sn[k] = base == 0 ? sn0[k] : 0.f;
      if (it < n) {
        xa[k] = src[(size_t)h * d + i];
        xb[k] = src[(size_t)h * d + i + half];
        if (base > 0 && h < nq + nkv) {
          cs[k] = rc[(size_t)pos * half + i];
          sn[k] = rsn[(size_t)pos * half + i];
        }
      }
    }
#pragma unroll
    for (int k = 0; k < RS_ITEMS; ++k) {
      const int it = base + k * RS_THREADS + threadIdx.x;
      const int hl = it / half, i = it - hl * half, h = h0 + hl;
      if (it >= n) continue;
      if (h >= nq + nkv) {   // value head: plain copy
        if (slot_ok) {
          T* v = vc + kv_row(page, seq, nkv, h - nq - nkv, cap, slot) * d;
          v[i] = Elem<T>::from_f(xa[k]);
          v[i + half] = Elem<T>::from_f(xb[k]);
        }
        continue;
      }
      if (h >= nq && !slot_ok) continue;
      float lo, hi;
      rope_pair(xa[k], xb[k], cs[k], sn[k], lo, hi);
      T* dst = h < nq ? q_out + ((size_t)r * nq + h) * d : kc + kv_row(page, seq, nkv, h - nq, cap, slot) * d;
      dst[i] = Elem<T>::from_f(lo);
      dst[i + half] = Elem<T>::from_f(hi);
    }
  }
}

int rope_store(cudaStream_t st, int dtype, const float* qkv, int R, int nq, int nkv, int d,
               const int* row_pos, const int* row_slot, const int* row_seq, const float* rope_cos,
               const float* rope_sin, void* q_out, void* kcache, void* vcache, int cap, int* err,
               int slot_limit, const KvPage& page) {
  if (R <= 0) return 0;
  // blocks of RS_HEADS heads of one row: a 7B verify pass (61 rows x 96 heads) is one wave
  // of resident blocks, so the next kernel can be scheduled while this one runs
  dim3 grid(R, (nq + 2 * nkv + RS_HEADS - 1) / RS_HEADS);
  const int threads = RS_THREADS;
  if (dtype == DT_F32)
    launch_k(rope_store_k<float>, grid, threads, 0, st, qkv, nq, nkv, d, row_pos, row_slot, row_seq, rope_cos, rope_sin,
                                                  (float*)q_out, (float*)kcache, (float*)vcache, cap, err, slot_limit, page);
  else
    launch_k(rope_store_k<__nv_bfloat16>, grid, threads, 0, st, qkv, nq, nkv, d, row_pos, row_slot, row_seq, rope_cos,
                                                          rope_sin, (__nv_bfloat16*)q_out, (__nv_bfloat16*)kcache,
                                                          (__nv_bfloat16*)vcache, cap, err, slot_limit, page);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

// h = silu(gate) * up over a 2D grid (row, 1024-element chunk), 4 elements per thread.
template <typename T>
__global__ void swiglu_k(const float* gu, int F, T* out) {
  PDL_ENTRY();
  const int r = blockIdx.x;
  const float* g = gu + (size_t)r * 2 * F;
  const int i0 = (blockIdx.y * blockDim.x + threadIdx.x) * 4;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int i = i0 + j;
    if (i < F) {
      if constexpr (std::is_same<T, __nv_bfloat16>::value) out[(size_t)r * F + i] = Elem<T>::from_f(silu_mul_bf16(g[i], g[F + i]));
      else out[(size_t)r * F + i] = Elem<T>::from_f(silu_mul(g[i], g[F + i]));
    }
  }
}

int swiglu_rows(cudaStream_t st, int dtype, const float* gu, int F, int R, void* out) {
  if (R <= 0) return 0;
  dim3 grid(R, (F + 1023) / 1024);
  if (dtype == DT_F32) launch_k(swiglu_k<float>, grid, 256, 0, st, gu, F, (float*)out);
  else launch_k(swiglu_k<__nv_bfloat16>, grid, 256, 0, st, gu, F, (__nv_bfloat16*)out);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

// EAGLE-1 drafter input row: [E[tok]; feature] (2H). Rows whose length and bases allow it
// move in 16-byte words, and every thread issues all its loads before its stores (a
// strided element loop paid one memory round trip per iteration).
constexpr int ROW_UNROLL = 4;

template <typename T>
__global__ void concat_k(const T* E, int V, int H, const int* tok, const T* feat, const int* feat_row, T* out,
                         int* err) {
  PDL_ENTRY();
  const int r = blockIdx.x;
  int t = tok[r];
  if (t < 0 || t >= V) {
    if (threadIdx.x == 0) latch_error(err, DEVERR_BOUNDS);
    t = 0;
  }
  const T* e = E + (size_t)t * H;
  const T* f = feat + (size_t)feat_row[r] * H;
  T* o = out + (size_t)r * 2 * H;
  constexpr int VW = 16 / sizeof(T);
  if (H % VW == 0 && ((reinterpret_cast<uintptr_t>(e) | reinterpret_cast<uintptr_t>(f) |
                       reinterpret_cast<uintptr_t>(o)) & 15) == 0) {
    const int n = H / VW;
    const uint4* ev = reinterpret_cast<const uint4*>(e);
    const uint4* fv = reinterpret_cast<const uint4*>(f);
    uint4* ov = reinterpret_cast<uint4*>(o);
    for (int base = 0; base < n; base += ROW_UNROLL * blockDim.x) {
      uint4 a[ROW_UNROLL], b[ROW_UNROLL];
#pragma unroll
      for (int k = 0; k < ROW_UNROLL; ++k) {
        const int i = base + k * blockDim.x + threadIdx.x;
        if (i < n) { a[k] = ev[i]; b[k] = fv[i]; }
      }
#pragma unroll
      for (int k = 0; k < ROW_UNROLL; ++k) {
        const int i = base + k * blockDim.x + threadIdx.x;
        if (i < n) { ov[i] = a[k]; ov[n + i] = b[k]; }
      }
    }
    return;
  }
  for (int base = 0; base < H; base += ROW_UNROLL * blockDim.x) {
    T a[ROW_UNROLL], b[ROW_UNROLL];
#pragma unroll
    for (int k = 0; k < ROW_UNROLL; ++k) {
      const int i = base + k * blockDim.x + threadIdx.x;
      if (i < H) { a[k] = e[i]; b[k] = f[i]; }
    }
#pragma unroll
    for (int k = 0; k < ROW_UNROLL; ++k) {
      const int i = base + k * blockDim.x + threadIdx.x;
      if (i < H) { o[i] = a[k]; o[H + i] = b[k]; }
    }
  }
}

int concat_emb_feat(cudaStream_t st, int dtype, const void* E, int V, int H, const int* tok, const void* feat,
                    const int* feat_row, int R, void* out, int* err) {
  if (R <= 0) return 0;
  if (dtype == DT_F32)
    launch_k(concat_k<float>, R, 256, 0, st, (const float*)E, V, H, tok, (const float*)feat, feat_row, (float*)out, err);
  else
    launch_k(concat_k<__nv_bfloat16>, R, 256, 0, st, (const __nv_bfloat16*)E, V, H, tok, (const __nv_bfloat16*)feat,
                                               feat_row, (__nv_bfloat16*)out, err);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

// Row conversions fp32 <-> storage type, ROW_UNROLL elements per thread and pass with
// all loads issued before the stores.
template <typename T>
__global__ void convert_k(const float* x, int H, T* out, int ldo) {
  PDL_ENTRY();
  const int r = blockIdx.x;
  const float* xr = x + (size_t)r * H;
  T* o = out + (size_t)r * ldo;
  for (int base = 0; base < H; base += ROW_UNROLL * blockDim.x) {
    float v[ROW_UNROLL];
#pragma unroll
    for (int k = 0; k < ROW_UNROLL; ++k) {
      const int i = base + k * blockDim.x + threadIdx.x;
      v[k] = i < H ? xr[i] : 0.f;
    }
#pragma unroll
    for (int k = 0; k < ROW_UNROLL; ++k) {
      const int i = base + k * blockDim.x + threadIdx.x;
      if (i < H) o[i] = Elem<T>::from_f(v[k]);
    }
  }
}

template <typename T>
__global__ void widen_k(const T* x, int ldx, int H, float* out) {
  PDL_ENTRY();
  const int r = blockIdx.x;
  const T* xr = x + (size_t)r * ldx;
  float* o = out + (size_t)r * H;
  for (int base = 0; base < H; base += ROW_UNROLL * blockDim.x) {
    float v[ROW_UNROLL];
#pragma unroll
    for (int k = 0; k < ROW_UNROLL; ++k) {
      const int i = base + k * blockDim.x + threadIdx.x;
      v[k] = i < H ? Elem<T>::to_f(xr[i]) : 0.f;
    }
#pragma unroll
    for (int k = 0; k < ROW_UNROLL; ++k) {
      const int i = base + k * blockDim.x + threadIdx.x;
      if (i < H) o[i] = v[k];
    }
  }
}

int widen_rows(cudaStream_t st, int dtype, const void* x, int ldx, int H, int R, float* out) {
  if (R <= 0) return 0;
  if (dtype == DT_F32) launch_k(widen_k<float>, R, 256, 0, st, (const float*)x, ldx, H, out);
  else launch_k(widen_k<__nv_bfloat16>, R, 256, 0, st, (const __nv_bfloat16*)x, ldx, H, out);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

int convert_rows(cudaStream_t st, int dtype, const float* x, int H, int R, void* out, int ldo) {
  if (R <= 0) return 0;
  if (dtype == DT_F32) launch_k(convert_k<float>, R, 256, 0, st, x, H, (float*)out, ldo);
  else launch_k(convert_k<__nv_bfloat16>, R, 256, 0, st, x, H, (__nv_bfloat16*)out, ldo);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

// dst row didx[r] <- src row sidx[r] (identity when an index is null); 16-byte words when aligned.
__global__ void gather_k(const uint8_t* src, size_t src_ld, const int* sidx, size_t row_bytes, uint8_t* dst,
                         size_t dst_ld, const int* didx, int src_rows, int* err) {
  PDL_ENTRY();
  const int r = blockIdx.x;
  const int si = sidx ? sidx[r] : r;
  if (src_rows > 0 && (si < 0 || si >= src_rows)) {   // an index from the caller's data (a token id)
    if (threadIdx.x == 0) latch_error(err, DEVERR_BOUNDS);
    return;
  }
  const uint8_t* s = src + (size_t)si * src_ld;
  uint8_t* d = dst + (size_t)(didx ? didx[r] : r) * dst_ld;
  if (((reinterpret_cast<uintptr_t>(s) | reinterpret_cast<uintptr_t>(d) | row_bytes) & 15) == 0) {
    for (size_t i = threadIdx.x; i < row_bytes / 16; i += blockDim.x)
      reinterpret_cast<uint4*>(d)[i] = reinterpret_cast<const uint4*>(s)[i];
  } else {
    for (size_t i = threadIdx.x; i < row_bytes; i += blockDim.x) d[i] = s[i];
  }
}

int gather_rows(cudaStream_t st, size_t row_bytes, const void* src, size_t src_ld, const int* idx, int R,
                void* dst, size_t dst_ld, const int* dst_idx, int src_rows, int* err) {
  if (R <= 0) return 0;
  launch_k(gather_k, R, 128, 0, st, (const uint8_t*)src, src_ld, idx, row_bytes, (uint8_t*)dst, dst_ld, dst_idx,
           src_rows, err);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace eagle
