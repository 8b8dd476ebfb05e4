// Layer chain: one persistent launch runs a short program of dependent steps of a decoder
// layer -- tcgen05 projection GEMMs and the row-wise ops between them (RMSNorm, SwiGLU,
// rotary embedding with the KV-cache write, conversions, embedding gathers) -- separated
// by grid-wide barriers, one CTA per SM under a cooperative launch.
//
// Why: at decode batch sizes every projection is a pure weight stream. Launched one by
// one, each pays a prologue, a first-load latency and a stream-K tail during which HBM
// idles, and the row ops between them run on an idle memory system. Here the TMA
// producer walks the weight tiles of ALL the program's GEMMs in order and never waits for
// a barrier: only the activation (B) half of a stage waits until the step that produces
// it is complete grid-wide. While the CTAs finish one projection's tail, pass a barrier
// and run a row op, the ring is already filling with the next projection's weights.
//
// Roles (192 threads), as in the single GEMM: warp 0 = TMA producer, warp 1 = MMA issuer
// and TMEM owner, warps 2-5 = GEMM epilogue and the row ops.
//
// Barrier protocol: bar[0] counts CTA arrivals. Every CTA arrives once at the end of each
// step except the last, and only after it has seen the previous barrier complete, so
// bar[0] >= s * G means every CTA has finished steps < s: step s may then read them. Data
// written inside the launch is read back through L2 (ld.global.cg) or by TMA after a proxy
// fence. The last CTA to leave resets bar[0] and bar[1] (its exit ticket) for the next
// launch. Every wait is bounded; a timeout latches an error and the CTA unwinds.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>

#include "chain.h"
#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"

namespace eagle {

EAGLE_DEV void fence_proxy_async() { asm volatile("fence.proxy.async;" ::: "memory"); }
// A step with fewer units than CTAs is split over its first U CTAs only, so that every
// CTA taking part holds at least one unit (the split-tile tickets count contributors).
EAGLE_DEV int step_ctas(long long U, int G) { return U < (long long)G ? (int)U : G; }

// The CTA's GEMM units in program order: step s (a GEMM), `left` units still to go in the
// CTA's stream-K range of that step, the current unit as k-block k of tile (tn, tt).
// Advanced incrementally, so the hot loops divide only when they enter a step.
struct UnitCursor {
  int s, left;
  int k, kb, tn, tt, tiles_t, gemm;
};

EAGLE_DEV void cursor_seek(const ChainArgs& a, UnitCursor& c, int from, int cta, int G) {
  for (int s = from; s < a.nsteps; ++s) {
    const ChainStep& st = a.s[s];
    if (st.kind != CH_GEMM) continue;
    const long long U = st.units;
    const int gs = step_ctas(U, G);
    if (cta >= gs) continue;
    const long long b = (long long)cta * U / gs, e = (long long)(cta + 1) * U / gs;
    if (b < e) {
      const long long tile = b / st.kb;
      c.s = s; c.left = (int)(e - b);
      c.kb = st.kb; c.tiles_t = st.tiles_t; c.gemm = st.gemm;
      c.k = (int)(b - tile * st.kb);
      c.tn = (int)(tile / st.tiles_t); c.tt = (int)(tile - (long long)c.tn * st.tiles_t);
      return;
    }
  }
  c.s = a.nsteps; c.left = 0;
}

// Move n (<= left) units forward.
EAGLE_DEV void cursor_advance(const ChainArgs& a, UnitCursor& c, int n, int cta, int G) {
  c.left -= n;
  if (c.left == 0) {
    cursor_seek(a, c, c.s + 1, cta, G);
    return;
  }
  c.k += n;
  while (c.k >= c.kb) {
    c.k -= c.kb;
    if (++c.tt == c.tiles_t) { c.tt = 0; ++c.tn; }
  }
}

// One chunk of CH accumulator columns (tokens) of feature row `row` of tile (tn, tt).
template <int CH>
EAGLE_DEV void chain_epi(const ChainStep& st, int M, int tn, int tt, int BN, int row, int c0, const float* v) {
  const int f = tn * 128 + row;
  if (f >= st.N) return;
  const int j0 = tt * BN + c0;
  if (st.epi == EPI_ADD_F32) {
    // residual update: all reads first (one round trip), then the writes
    float* o = reinterpret_cast<float*>(st.out) + (size_t)j0 * st.ldo + f;
    float old[CH];
#pragma unroll
    for (int i = 0; i < CH; ++i) old[i] = (j0 + i < M) ? __ldcg(o + (size_t)i * st.ldo) : 0.f;
#pragma unroll
    for (int i = 0; i < CH; ++i)
      if (j0 + i < M) o[(size_t)i * st.ldo] = old[i] + v[i];
    return;
  }
#pragma unroll
  for (int i = 0; i < CH; ++i) {
    const int j = j0 + i;
    if (j < M) {
      const size_t o = (size_t)j * st.ldo + f;
      if (st.epi == EPI_F32) reinterpret_cast<float*>(st.out)[o] = v[i];
      else reinterpret_cast<__nv_bfloat16*>(st.out)[o] = __float2bfloat16_rn(v[i]);
    }
  }
}

EAGLE_DEV void store4(__nv_bfloat16* p, float x, float y, float z, float w) {
  __nv_bfloat162* q = reinterpret_cast<__nv_bfloat162*>(p);
  q[0] = __floats2bfloat162_rn(x, y);
  q[1] = __floats2bfloat162_rn(z, w);
}

// ---- row ops: 128 threads per CTA (tid), G CTAs. Kept out of line so their registers do
// not add to the GEMM roles' live ranges. ------------------------------------------------
EAGLE_DEV float load_in(const ChainStep& st, size_t i) {
  return st.in_bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(st.in)[i])
                    : __ldcg(reinterpret_cast<const float*>(st.in) + i);
}

// out = in * rsqrt(mean(in^2) + eps) * g, one row per CTA at a time; per-thread sums in
// index order, then a fixed warp / block tree.
// Rows of up to 128 * 4 * RN_V elements (fp32, H % 4 == 0) are read in one round of
// vector loads and kept in registers; others take a two-pass loop.
constexpr int RN_V = 10;

__device__ __noinline__ void row_rmsnorm(const ChainStep& st, int M, int cta, int G, int tid, float* red) {
  const __nv_bfloat16* g = reinterpret_cast<const __nv_bfloat16*>(st.aux);
  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(st.out);
  const bool vec = !st.in_bf16 && st.H % 4 == 0 && st.ldi % 4 == 0 && st.ldo % 4 == 0 && st.H <= 128 * 4 * RN_V;
  for (int r = cta; r < M; r += G) {
    const size_t base = (size_t)r * st.ldi;
    float s = 0.f;
    float4 xv[RN_V];
    uint2 gv[RN_V];
    if (vec) {
      const float* xr = reinterpret_cast<const float*>(st.in) + base;
#pragma unroll
      for (int j = 0; j < RN_V; ++j) {
        const int i = (j * 128 + tid) * 4;
        if (i < st.H) {
          xv[j] = __ldcg(reinterpret_cast<const float4*>(xr + i));
          gv[j] = *reinterpret_cast<const uint2*>(g + i);
        }
      }
#pragma unroll
      for (int j = 0; j < RN_V; ++j)
        if ((j * 128 + tid) * 4 < st.H) s += (xv[j].x * xv[j].x + xv[j].y * xv[j].y) + (xv[j].z * xv[j].z + xv[j].w * xv[j].w);
    } else {
#pragma unroll 8
      for (int i = tid; i < st.H; i += 128) {
        const float v = load_in(st, base + i);
        s += v * v;
      }
    }
    s = warp_sum(s);
    if ((tid & 31) == 0) red[tid >> 5] = s;
    named_bar_sync(1, 128);
    const float tot = (red[0] + red[1]) + (red[2] + red[3]);
    named_bar_sync(1, 128);
    const float rs = rsqrtf(tot / (float)st.H + st.eps);
    if (vec) {
#pragma unroll
      for (int j = 0; j < RN_V; ++j) {
        const int i = (j * 128 + tid) * 4;
        if (i < st.H) {
          const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&gv[j]);
          const float2 g01 = __bfloat1622float2(g2[0]), g23 = __bfloat1622float2(g2[1]);
          __nv_bfloat162 o[2] = {__floats2bfloat162_rn(xv[j].x * rs * g01.x, xv[j].y * rs * g01.y),
                                 __floats2bfloat162_rn(xv[j].z * rs * g23.x, xv[j].w * rs * g23.y)};
          *reinterpret_cast<uint2*>(out + (size_t)r * st.ldo + i) = *reinterpret_cast<const uint2*>(o);
        }
      }
    } else {
#pragma unroll 8
      for (int i = tid; i < st.H; i += 128)
        out[(size_t)r * st.ldo + i] = __float2bfloat16_rn(load_in(st, base + i) * rs * __bfloat162float(g[i]));
    }
  }
}

// 4 consecutive features per item (F % 4 == 0, so rows of gu stay 16-byte aligned), four
// items in flight per thread.

__device__ __noinline__ void row_swiglu(const ChainStep& st, int M, int t0, int stride) {
  const float* gu = reinterpret_cast<const float*>(st.in);
  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(st.out);
  const int F = st.H, F4 = F / 4, n = M * F4;
  constexpr int SB = 4;
  for (int i0 = t0; i0 < n; i0 += SB * stride) {
    float4 g[SB], u[SB];
    int off[SB];
#pragma unroll
    for (int q = 0; q < SB; ++q) {
      const int i = i0 + q * stride;
      if (i < n) {
        const int r = i / F4, c = (i - r * F4) * 4;
        off[q] = r * F + c;
        g[q] = __ldcg(reinterpret_cast<const float4*>(gu + (size_t)r * 2 * F + c));
        u[q] = __ldcg(reinterpret_cast<const float4*>(gu + (size_t)r * 2 * F + F + c));
      }
    }
#pragma unroll
    for (int q = 0; q < SB; ++q) {
      if (i0 + q * stride < n) {
        __nv_bfloat162* o = reinterpret_cast<__nv_bfloat162*>(out + off[q]);
        o[0] = __floats2bfloat162_rn(silu_mul_bf16(g[q].x, u[q].x), silu_mul_bf16(g[q].y, u[q].y));
        o[1] = __floats2bfloat162_rn(silu_mul_bf16(g[q].z, u[q].z), silu_mul_bf16(g[q].w, u[q].w));
      }
    }
  }
}

__device__ __noinline__ void row_convert(const ChainStep& st, int M, int t0, int stride) {
  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(st.out);
  const float* in = reinterpret_cast<const float*>(st.in);
  const int H4 = st.H / 4, n = M * H4;
  for (int i = t0; i < n; i += stride) {
    const int r = i / H4, c = (i - r * H4) * 4;
    const float4 v = __ldcg(reinterpret_cast<const float4*>(in + (size_t)r * st.ldi + c));
    store4(out + (size_t)r * st.ldo + c, v.x, v.y, v.z, v.w);
  }
}

__device__ __noinline__ void row_embed(const ChainStep& st, int M, int t0, int stride, int* err) {
  const __nv_bfloat16* E = reinterpret_cast<const __nv_bfloat16*>(st.aux);
  float* out = reinterpret_cast<float*>(st.out);
  const int H = st.H, n = M * H;
  for (int i = t0; i < n; i += stride) {
    const int r = i / H, c = i - r * H;
    int t = st.idx[r];
    if (t < 0 || t >= st.V) {
      if (c == 0) latch_error(err, DEVERR_BOUNDS);
      t = 0;
    }
    out[i] = __bfloat162float(E[(size_t)t * H + c]);
  }
}

// [E[idx[r]] ; feat[idx2[r]]] -> out [M][2H] (bf16)
__device__ __noinline__ void row_concat(const ChainStep& st, int M, int t0, int stride, int* err) {
  const __nv_bfloat16* E = reinterpret_cast<const __nv_bfloat16*>(st.aux);
  const __nv_bfloat16* feat = reinterpret_cast<const __nv_bfloat16*>(st.in);
  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(st.out);
  const int H = st.H, n = M * 2 * H;
  for (int i = t0; i < n; i += stride) {
    const int r = i / (2 * H), c = i - r * 2 * H;
    if (c < H) {
      int t = st.idx[r];
      if (t < 0 || t >= st.V) {
        if (c == 0) latch_error(err, DEVERR_BOUNDS);
        t = 0;
      }
      out[i] = E[(size_t)t * H + c];
    } else {
      out[i] = feat[(size_t)st.idx2[r] * H + (c - H)];
    }
  }
}

// Rotate-half RoPE on the q and k heads of the fused [q | k | v] projection; q to its
// buffer, k and v into the cache at the row's slot (a slot outside [0, cap) latches a
// capacity error and skips the cache write). Items of 4 consecutive elements (d % 8 == 0).

__device__ __noinline__ void row_rope(const ChainRope& p, int M, int t0, int stride, int* err) {
  const int half = p.d / 2, h4 = half / 4, d4 = p.d / 4;
  const int rot = (p.nq + p.nkv) * h4;
  const int per_row = rot + p.nkv * d4;
  const int n = M * per_row;
  const int ld = (p.nq + 2 * p.nkv) * p.d;
  __nv_bfloat16* q = reinterpret_cast<__nv_bfloat16*>(p.q);
  __nv_bfloat16* kc = reinterpret_cast<__nv_bfloat16*>(p.kc);
  __nv_bfloat16* vc = reinterpret_cast<__nv_bfloat16*>(p.vc);
  // two items per turn: all loads of both are issued before any store
  for (int i0 = t0; i0 < n; i0 += 2 * stride) {
    int r[2], j[2], slot[2], seq[2], pos[2];
    float4 x0[2], x1[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int i = i0 + u * stride;
      r[u] = -1;
      if (i >= n) continue;
      r[u] = i / per_row;
      j[u] = i - r[u] * per_row;
      slot[u] = p.slot[r[u]];
      seq[u] = p.seq[r[u]];
      pos[u] = p.pos[r[u]];
      const float* src = p.qkv + (size_t)r[u] * ld;
      int c0, c1 = -1;
      if (j[u] < rot) {
        const int h = j[u] / h4, e = (j[u] - h * h4) * 4;
        c0 = h * p.d + e;
        c1 = c0 + half;
      } else {
        const int jj = j[u] - rot;
        const int h = jj / d4, e = (jj - h * d4) * 4;
        c0 = (p.nq + p.nkv + h) * p.d + e;
      }
      x0[u] = __ldcg(reinterpret_cast<const float4*>(src + c0));
      if (c1 >= 0) x1[u] = __ldcg(reinterpret_cast<const float4*>(src + c1));
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (r[u] < 0) continue;
      const bool slot_ok = slot[u] >= 0 && slot[u] < p.cap;
      if (j[u] < rot) {
        const int h = j[u] / h4, e = (j[u] - h * h4) * 4;
        if (h >= p.nq && !slot_ok) {
          if (e == 0) latch_error(err, DEVERR_CAPACITY);
          continue;
        }
        const float4 c = *reinterpret_cast<const float4*>(p.cos + (size_t)pos[u] * half + e);
        const float4 sn = *reinterpret_cast<const float4*>(p.sin + (size_t)pos[u] * half + e);
        const float4 a = x0[u], b = x1[u];
        __nv_bfloat16* dst = h < p.nq ? q + ((size_t)r[u] * p.nq + h) * p.d
                                      : kc + ((size_t)(seq[u] * p.nkv + (h - p.nq)) * p.cap + slot[u]) * p.d;
        float l0, l1, l2, l3, h0, h1, h2, h3;
        rope_pair(a.x, b.x, c.x, sn.x, l0, h0);
        rope_pair(a.y, b.y, c.y, sn.y, l1, h1);
        rope_pair(a.z, b.z, c.z, sn.z, l2, h2);
        rope_pair(a.w, b.w, c.w, sn.w, l3, h3);
        store4(dst + e, l0, l1, l2, l3);
        store4(dst + e + half, h0, h1, h2, h3);
      } else {
        if (!slot_ok) continue;
        const int jj = j[u] - rot;
        const int h = jj / d4, e = (jj - h * d4) * 4;
        store4(vc + ((size_t)(seq[u] * p.nkv + h) * p.cap + slot[u]) * p.d + e, x0[u].x, x0[u].y, x0[u].z,
               x0[u].w);
      }
    }
  }
}

template <int BN>
__global__ void __launch_bounds__(192, 1)
    chain_k(const __grid_constant__ ChainMaps maps, const __grid_constant__ ChainArgs a) {
  using C = TcCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* staging = reinterpret_cast<float*>(smem + C::STAGES * C::STAGE);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE + C::STAGING);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::STAGES;
  uint64_t* tfull = bars + 2 * C::STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* bcast = reinterpret_cast<volatile int*>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, cta = blockIdx.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(smem_u32(full + s), 1);
      mbar_init(smem_u32(empty + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(tfull + b), 1);
      mbar_init(smem_u32(tempty + b), 128);
    }
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
  pdl_trigger();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // Two cursors over the same unit sequence: A (weights) runs ahead as far as the ring
      // allows; B (activations) follows once the unit's step is open.
      const uint64_t pol_w = l2_policy_evict_first();
      const uint64_t pol_x = l2_policy_evict_last();
      UnitCursor ca, cb;
      cursor_seek(a, ca, 0, cta, G);
      cb = ca;
      uint32_t nA = 0, nB = 0;      // units armed (A issued) / completed with their B half
      int slotA = 0, slotB = 0;
      uint32_t phA = 0;
      int open = -1;          // steps <= open may be read
      uint64_t idle_since = 0;
      bool idle = false;
      uint32_t spins = 0;
      while (cb.s < a.nsteps) {
        bool prog = false;
        if (ca.s < a.nsteps) {
          if (mbar_try(smem_u32(empty + slotA), phA ^ 1u)) {
            const uint32_t fb = smem_u32(full + slotA);
            mbar_expect_tx(fb, C::STAGE);
            tma_load_2d(smem_u32(smem + slotA * C::STAGE), &maps.w[ca.gemm], ca.k * 64, ca.tn * 128, fb, pol_w);
            cursor_advance(a, ca, 1, cta, G);
            ++nA;
            if (++slotA == C::STAGES) { slotA = 0; phA ^= 1u; }
            prog = true;
          }
        }
        if (nB < nA) {
          const int s = cb.s;
          if (s > open) {
            if (open < 0) {   // the previous grid's outputs (and its reset of bar) first
              pdl_wait();
              open = 0;
            }
            if (s > open) {
              const unsigned v = ld_acquire_u32(a.bar);
              if (v >= (unsigned)s * (unsigned)G) open = (int)(v / (unsigned)G);
            }
            if (s <= open) {   // acquire, then order it before this thread's TMA reads
              fence_acq_rel_gpu();
              fence_proxy_async();
            }
          }
          if (s <= open) {
            tma_load_2d(smem_u32(smem + slotB * C::STAGE) + C::A_BYTES, &maps.x[cb.gemm], cb.k * 64, cb.tt * BN,
                        smem_u32(full + slotB), pol_x);
            cursor_advance(a, cb, 1, cta, G);
            ++nB;
            if (++slotB == C::STAGES) slotB = 0;
            prog = true;
          }
        }
        if (prog) {
          idle = false;
        } else if (nB == nA && ca.s < a.nsteps) {
          // streaming: every armed stage has its activations; sleep on the next slot
          if (!mbar_wait(smem_u32(empty + slotA), phA ^ 1u, abort_flag, a.err)) break;
        } else {
          // waiting for a step to open (polled above): look at the shared error word now
          // and then only, so the poll itself stays the one global access per turn
          if (*abort_flag || ((++spins & 255u) == 0 && err_raised(a.err))) { *abort_flag = 1; break; }
          const uint64_t now = globaltimer();
          if (!idle) { idle = true; idle_since = now; }
          else if (now - idle_since > EAGLE_WAIT_LIMIT_NS) {
            *abort_flag = 1;
            latch_error(a.err, DEVERR_MBAR_TIMEOUT);
            break;
          }
        }
      }
      if (*abort_flag) {
        // complete every stage already armed (its B half may still be missing), then wait
        // for the copies in flight so none lands after the CTA has left
        while (nB < nA) {
          tma_load_2d(smem_u32(smem + slotB * C::STAGE) + C::A_BYTES, &maps.x[cb.gemm], cb.k * 64, cb.tt * BN,
                      smem_u32(full + slotB), pol_x);
          cursor_advance(a, cb, 1, cta, G);
          ++nB;
          if (++slotB == C::STAGES) slotB = 0;
        }
        for (uint32_t j = nA > (uint32_t)C::STAGES ? nA - C::STAGES : 0; j < nA; ++j)
          mbar_wait(smem_u32(full + (int)(j % C::STAGES)), (j / C::STAGES) & 1u, abort_flag, a.err, false);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t IDESC = idesc_bf16<BN>();
      UnitCursor c;
      cursor_seek(a, c, 0, cta, G);
      int slot = 0;
      uint32_t ph = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      while (ok && c.s < a.nsteps) {
        const int seg = min(c.left, c.kb - c.k);   // units of this tile in the CTA's range
        if (!mbar_wait(smem_u32(tempty + acc), acc_phase ^ 1, abort_flag, a.err)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * BN);
        for (int i = 0; i < seg; ++i) {
          if (!mbar_wait(smem_u32(full + slot), ph, abort_flag, a.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + slot * C::STAGE);
          const uint64_t da = sdesc_sw128(sa), db = sdesc_sw128(sa + C::A_BYTES);
#pragma unroll
          for (int k = 0; k < 4; ++k) tc_mma_bf16(d, da + 2 * k, db + 2 * k, IDESC, (i || k) ? 1u : 0u);
          tc_commit(smem_u32(empty + slot));
          if (++slot == C::STAGES) { slot = 0; ph ^= 1u; }
        }
        if (!ok) break;
        tc_commit(smem_u32(tfull + acc));
        acc ^= 1;
        if (!acc) acc_phase ^= 1;
        cursor_advance(a, c, seg, cta, G);
      }
      if (!ok) {
        tc_commit(smem_u32(drain));
        mbar_wait(smem_u32(drain), 0, abort_flag, a.err, false);
      }
    }
  } else {
    pdl_wait();
    const int tid = threadIdx.x - 64;
    const int ew = warp - 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const bool leader = (ew == 0 && lane == 0);
    const int t0 = cta * 128 + tid, tstride = G * 128;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int s = 0; s < a.nsteps; ++s) {
      const ChainStep& st = a.s[s];
      if (st.kind == CH_GEMM) {
        const long long U = st.units;
        const int gs = step_ctas(U, G);
        const long long u_begin = cta < gs ? (long long)cta * U / gs : 0;
        const long long u_end = cta < gs ? (long long)(cta + 1) * U / gs : 0;
        const long long first_tile = u_begin / st.kb;
        bool ok = true;
        for (long long u = u_begin; u < u_end;) {
          const long long tile = u / st.kb;
          const long long seg_end = min(u_end, (tile + 1) * st.kb);
          const bool whole = (u == tile * st.kb) && (seg_end == (tile + 1) * st.kb);
          const int tn = (int)(tile / st.tiles_t), tt = (int)(tile % st.tiles_t);
          if (leader) bcast[0] = mbar_wait(smem_u32(tfull + acc), acc_phase, abort_flag, a.err) ? 1 : 0;
          named_bar_sync(1, 128);
          ok = bcast[0] != 0;
          named_bar_sync(1, 128);
          if (!ok) break;
          tc_fence_after();
          const uint32_t tb = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
          if (whole) {
            for (int c0 = 0; c0 < BN; c0 += C::CH) {
              float v[C::CH];
              if constexpr (C::CH == 32) tmem_ld32(tb + c0, v); else tmem_ld16(tb + c0, v);
              chain_epi<C::CH>(st, a.M, tn, tt, BN, row, c0, v);
            }
            tc_fence_before();
            mbar_arrive(smem_u32(tempty + acc));
          } else {
            const int slot = (tile == first_tile) ? 0 : 1;
            float* part = a.partials + (size_t)(cta * 2 + slot) * BN * 128;
            for (int c0 = 0; c0 < BN; c0 += C::CH) {
              float v[C::CH];
              if constexpr (C::CH == 32) tmem_ld32(tb + c0, v); else tmem_ld16(tb + c0, v);
#pragma unroll
              for (int i = 0; i < C::CH; ++i) part[(c0 + i) * 128 + row] = v[i];
            }
            tc_fence_before();
            mbar_arrive(smem_u32(tempty + acc));
            // publish the partial: every thread fences, the CTA synchronises, one thread
            // takes the tile's ticket between gpu-scope fences; the last contributor sums
            // the partials in contributor order (two contributors' loads in flight)
            __threadfence();
            named_bar_sync(1, 128);
            const int cf = cta_of_unit(tile * st.kb, U, gs);
            const int cl = cta_of_unit((tile + 1) * st.kb - 1, U, gs);
            if (leader) {
              __threadfence();
              const int old = atomicAdd(a.counters + tile, 1);
              bcast[1] = (old == cl - cf) ? 1 : 0;
              __threadfence();
            }
            named_bar_sync(1, 128);
            if (bcast[1]) {
              __threadfence();
              // every contributor after the first began its range inside this tile (slot 0)
              const int s_first = ((long long)cf * U / gs < tile * st.kb) ? 1 : 0;
              for (int c0 = 0; c0 < BN; c0 += C::CH) {
                float v[C::CH];
#pragma unroll
                for (int i = 0; i < C::CH; ++i) v[i] = 0.f;
                for (int cc = cf; cc <= cl; cc += 2) {
                  const bool two = cc + 1 <= cl;
                  const float* p0 = a.partials + (size_t)(cc * 2 + (cc == cf ? s_first : 0)) * BN * 128 + c0 * 128 + row;
                  const float* p1 = a.partials + (size_t)((cc + 1) * 2) * BN * 128 + c0 * 128 + row;
                  float x0[C::CH], x1[C::CH];
#pragma unroll
                  for (int i = 0; i < C::CH; ++i) {
                    x0[i] = __ldcg(p0 + i * 128);
                    x1[i] = two ? __ldcg(p1 + i * 128) : 0.f;
                  }
#pragma unroll
                  for (int i = 0; i < C::CH; ++i) v[i] += x0[i];
                  if (two) {
#pragma unroll
                    for (int i = 0; i < C::CH; ++i) v[i] += x1[i];
                  }
                }
                chain_epi<C::CH>(st, a.M, tn, tt, BN, row, c0, v);
              }
              if (leader) a.counters[tile] = 0;
            }
            named_bar_sync(1, 128);
          }
          u = seg_end;
          acc ^= 1;
          if (!acc) acc_phase ^= 1;
        }
        if (!ok) break;
      } else {
        if (s > 0) {
          if (leader) {
            bcast[0] = grid_wait(a.bar, (unsigned)s * (unsigned)G, abort_flag, a.err) ? 1 : 0;
            fence_acq_rel_gpu();
          }
          named_bar_sync(1, 128);
          const bool ok = bcast[0] != 0;
          named_bar_sync(1, 128);
          if (!ok) break;
        }
        switch (st.kind) {
          case CH_RMSNORM: row_rmsnorm(st, a.M, cta, G, tid, staging); break;
          case CH_SWIGLU: row_swiglu(st, a.M, t0, tstride); break;
          case CH_ROPE: row_rope(a.rope, a.M, t0, tstride, a.err); break;
          case CH_CONVERT: row_convert(st, a.M, t0, tstride); break;
          case CH_EMBED: row_embed(st, a.M, t0, tstride, a.err); break;
          case CH_CONCAT: row_concat(st, a.M, t0, tstride, a.err); break;
          default: break;
        }
      }
      if (s + 1 < a.nsteps) {
        // release: every thread fences its writes at gpu scope and orders them for the
        // async proxy (TMA readers), the CTA synchronises, then one thread publishes
        __threadfence();
        fence_proxy_async();
        named_bar_sync(1, 128);
        if (leader) {
          // a CTA arrives at barrier s only after barrier s - 1 has completed: a CTA with no
          // units in a GEMM step would otherwise run ahead and add a second arrival before
          // the slow CTAs of step s - 1 have arrived, opening step s + 1 early
          const bool ok = !(s > 0 && st.kind == CH_GEMM) || grid_wait(a.bar, (unsigned)s * (unsigned)G, abort_flag, a.err);
          if (ok) {
            __threadfence();
            red_release_add(a.bar, 1u);
          }
          bcast[1] = ok ? 1 : 0;
        }
        named_bar_sync(1, 128);
        const bool arrived = bcast[1] != 0;
        named_bar_sync(1, 128);
        if (!arrived) break;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(a.bar + 1, 1u) == (unsigned)G - 1) {
      atomicExch(a.bar, 0u);
      atomicExch(a.bar + 1, 0u);
    }
  }
}

// ---- host side ----------------------------------------------------------------------------------
static int chain_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n > num_sms_cap()) n = num_sms_cap();
    if (n <= 0) n = 1;
  }
  return n;
}

template <int BN>
static cudaError_t chain_launch_bn(cudaStream_t st, const ChainMaps& maps, const ChainArgs& a) {
  using C = TcCfg<BN>;
  static bool attr = false;
  static bool pdl_ok = true;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(chain_k<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, chain_k<BN>, 192, C::SMEM);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    attr = true;
  }
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeCooperative;
  at[0].val.cooperative = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(chain_sms());
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = st;
  cfg.attrs = at;
  cfg.numAttrs = (pdl_ok && pdl_enabled()) ? 2 : 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, chain_k<BN>, maps, a);
  if (e != cudaSuccess && cfg.numAttrs == 2) {
    // cooperative launches that refuse the programmatic-serialization attribute run without it
    cudaGetLastError();
    pdl_ok = false;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, chain_k<BN>, maps, a);
  }
  return e;
}

static_assert(sizeof(ChainArgs) + sizeof(ChainMaps) <= 4000, "chain kernel parameters exceed 4 KB");

int chain_run(cudaStream_t st, const ChainProgram& p) {
  if (p.M <= 0 || p.nsteps <= 0 || p.nsteps > CHAIN_MAX_STEPS || !p.bar || !p.partials || !p.counters) return -1;
  const int BN = gemm_bn_for(p.M);
  const int G = chain_sms();
  ChainMaps maps;
  memset(&maps, 0, sizeof(maps));
  ChainArgs a = p.args;
  a.nsteps = p.nsteps;
  a.M = p.M;
  a.partials = p.partials;
  a.counters = p.counters;
  a.bar = p.bar;
  a.err = p.err;
  auto aligned16 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15) == 0; };
  int ng = 0;
  for (int s = 0; s < p.nsteps; ++s) {
    ChainStep& c = a.s[s];
    // row ops index elements with 32-bit integers
    const long long w = c.kind == CH_ROPE ? (long long)(a.rope.nq + 2 * a.rope.nkv) * a.rope.d : 2LL * c.H;
    if ((long long)p.M * w >= (1LL << 31)) return -1;
    if (c.kind == CH_SWIGLU && (c.H % 4 || !aligned16(c.in) || !aligned16(c.out))) return -1;
    if (c.kind == CH_ROPE && (a.rope.d % 8 || !aligned16(a.rope.qkv))) return -1;
    if (c.kind == CH_CONVERT && (c.H % 4 || c.ldi % 4 || c.ldo % 4 || !aligned16(c.in))) return -1;
    if (c.kind != CH_GEMM) continue;
    if (ng >= CHAIN_MAX_GEMMS) return -1;
    const ChainGemm& g = p.gemm[s];
    if (!g.W || !g.X || c.K % 8 || !aligned16(g.W) || !aligned16(g.X) || !aligned16(c.out)) return -1;
    if (c.epi != EPI_F32 && c.epi != EPI_BF16 && c.epi != EPI_ADD_F32) return -1;
    if (!make_tmap_bf16(&maps.w[ng], g.W, c.N, c.K, 128)) return -3;
    if (!make_tmap_bf16(&maps.x[ng], g.X, p.M, c.K, BN, g.ldx)) return -3;
    c.gemm = ng++;
    c.tiles_t = (p.M + BN - 1) / BN;
    c.kb = (c.K + 63) / 64;
    c.units = (long long)((c.N + 127) / 128) * c.tiles_t * c.kb;
    if (c.units * G >= (1LL << 31) || c.units / c.kb > p.counters_len) return -2;
  }
  cudaError_t e;
  switch (BN) {
    case 16: e = chain_launch_bn<16>(st, maps, a); break;
    case 32: e = chain_launch_bn<32>(st, maps, a); break;
    case 64: e = chain_launch_bn<64>(st, maps, a); break;
    case 128: e = chain_launch_bn<128>(st, maps, a); break;
    default: e = chain_launch_bn<256>(st, maps, a); break;
  }
  return e == cudaSuccess ? 0 : -4;
}

}  // namespace eagle
