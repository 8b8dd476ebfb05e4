// bf16 weight-streaming GEMM on the 5th-generation tensor cores (tcgen05 + TMA + TMEM).
//
//   Y[M][N] = X[M][K] * W[N][K]^T      (X: activations/tokens, W: nn.Linear-layout weight)
//
// Decode-time projections are skinny (M = 1..61 tokens at batch 1), so the weight is the
// 128-row "A" operand of tcgen05.mma and the tokens are the N-side operand (BN = 16..256
// columns, zero-filled by TMA past M). The accumulator tile D[128 features][BN tokens]
// lives in TMEM, double-buffered so the epilogue of one tile overlaps the next tile's
// main loop.
//
// Work split: stream-K over the (weight tile, k-block) units of one token tile, cut into
// gridDim.x equal contiguous ranges, one per persistent CTA, so every SM streams the same
// number of weight bytes whatever the shape. The ranges depend on (N, K, SM count) only,
// never on the number of tokens M: with several token tiles (M > 256) each CTA runs its
// range once per token tile, segment by segment (a segment = the range's piece of one
// weight tile, run for every token tile before the next, so the token tiles re-read its
// weight boxes from L2). Every output element is therefore summed over the same k-split
// points in the same order whatever M is, and a token's projection is bit-identical in a
// 1-row and a 1088-row GEMM. Shapes with fewer weight tiles than CTAs and several token
// tiles take the whole-tile schedule below instead, which adds the same pieces in the same
// order inside one CTA. A tile split across CTAs is finished by its first
// contributor, for which it is the last segment of its range: the later contributors reach
// the tile at the start of their ranges, publish fp32 partials and count themselves in on
// a per-(tile, token tile) counter; the owner waits (bounded) for that count and adds the
// partials to its own accumulator in contributor order, so results do not depend on timing
// and the owner never writes its own partial. A contributor publishes before it waits on
// anything and every CTA of the grid is resident at once (one CTA per SM, at most one per
// SM launched), so the wait always ends.
//
// Roles (192 threads): warp 0 = TMA producer, warp 1 = MMA issuer and TMEM owner,
// warps 2-5 = epilogue (TMEM -> registers -> global / fused LM-head reduction).
// Every mbarrier wait is bounded; on a timeout the CTA latches an error, drains its
// in-flight copies and MMAs, frees TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <map>
#include <mutex>
#include <tuple>
#include <utility>

#include "common.cuh"
#include "kernels.h"
#include "lmhead.cuh"
#include "tc_common.cuh"

namespace eagle {

struct GemmArgs {
  int M, N, K;
  int tiles_t;        // token tiles
  int kb;             // 64-wide k-blocks
  long long units;    // units of one token tile: tiles_n * kb
  int epi;
  void* out;
  int ldo;
  float* partials;
  int* counters;
  int* err;
  HeadParams head;
  QkvEpi qkv;
};


// Epilogue variants, one kernel instantiation each: generic (store / residual add / fused LM
// head, chosen by a.epi), SwiGLU of [gate; up] tile pairs, RoPE + KV-cache write of QKV.
enum { MODE_GENERIC = 0, MODE_QKV = 1, MODE_SWIGLU = 2 };

template <int CH, int MODE>
__device__ __forceinline__ void epi_chunk(const GemmArgs& a, int tn, int tt, int BN, int row, int c0,
                                          const float* v, float* staging, int ew, int lane) {
  if constexpr (MODE == MODE_SWIGLU) {
    // accumulator rows 0-63: gate features tn*64.., rows 64-127: the matching up features.
    if (a.epi == EPI_GU) {
      // fp32 gate and up values to out [M][2N] (gate at f, up at N + f), for a separate
      // SwiGLU pass that then sees exactly the values the fused epilogue would
      const int f = tn * 64 + (row & 63);
      if (f < a.N) {
        float* o = reinterpret_cast<float*>(a.out) + (row < 64 ? f : a.N + f);
#pragma unroll
        for (int i = 0; i < CH; ++i) {
          const int j = tt * BN + c0 + i;
          if (j < a.M) o[(size_t)j * a.ldo] = v[i];
        }
      }
      return;
    }
    // Through shared memory every thread then takes one gate/up pair for half the columns.
#pragma unroll
    for (int i = 0; i < CH; ++i) staging[i * 128 + row] = v[i];
    named_bar_sync(2, 128);
    const int r = row & 63, c_lo = (row >> 6) * (CH / 2);
    const int f = tn * 64 + r;
    if (f < a.N) {
      __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(a.out);
#pragma unroll
      for (int i = 0; i < CH / 2; ++i) {
        const int c = c_lo + i;
        const int j = tt * BN + c0 + c;
        if (j < a.M)
          o[(size_t)j * a.ldo + f] = __float2bfloat16_rn(silu_mul_bf16(staging[c * 128 + r], staging[c * 128 + 64 + r]));
      }
    }
    named_bar_sync(2, 128);
    return;
  }
  if constexpr (MODE == MODE_QKV) {
    // 16-column chunks. Shared memory holds the chunk's values [16][128], the cos/sin rows
    // of its positions [16][d/2] each, and the tile's per-column slot / sequence / position.
    // The code stays short (rolled loops): it runs cold at the end of the kernel.
    static_assert(CH == 16, "the QKV epilogue works on 16-column chunks");
    const QkvEpi& q = a.qkv;
    int* meta = reinterpret_cast<int*>(staging + 32 * 128);
    float* css = staging + CH * 128;
    float* sns = css + CH * 64;
    const int d = q.d, half = d >> 1, hs = __ffs(half) - 1;
    if (c0 == 0) {
      for (int t = row; t < BN; t += 128) {
        const int j = min(tt * BN + t, a.M - 1);
        meta[t] = q.slot[j];
        meta[256 + t] = q.seq[j];
        meta[512 + t] = q.pos[j];
      }
      named_bar_sync(2, 128);
    }
#pragma unroll
    for (int i = 0; i < CH; ++i) staging[i * 128 + row] = v[i];
#pragma unroll
    for (int k = 0; k < CH * 64 / 128; ++k) {
      const int idx = k * 128 + row;
      if (idx < (CH << hs)) {
        const int ci = meta[512 + c0 + (idx >> hs)] * half + (idx & (half - 1));
        css[idx] = q.cos[ci];
        sns[idx] = q.sin[ci];
      }
    }
    named_bar_sync(2, 128);
    const int f = tn * 128 + row;
    if (f < a.N) {
      const int h = f >> (hs + 1), e = f & (d - 1);
      const bool lo_half = e < half;
      const int prow = lo_half ? row + half : row - half;
      const int eh = e & (half - 1);
      const int jn = min(CH, a.M - (tt * BN + c0));
      if (h < q.nq + q.nkv) {
        __nv_bfloat16* qo = reinterpret_cast<__nv_bfloat16*>(q.q);
        __nv_bfloat16* ko = reinterpret_cast<__nv_bfloat16*>(q.kc);
#pragma unroll 4
        for (int i = 0; i < jn; ++i) {
          const int j = tt * BN + c0 + i;
          const float x = staging[i * 128 + row], y = staging[i * 128 + prow];
          const float c = css[(i << hs) + eh], sn = sns[(i << hs) + eh];
          float lo, hi;
          if (lo_half) rope_pair(x, y, c, sn, lo, hi);
          else rope_pair(y, x, c, sn, lo, hi);
          const __nv_bfloat16 r = __float2bfloat16_rn(lo_half ? lo : hi);
          if (h < q.nq) {
            qo[((size_t)j * q.nq + h) * d + e] = r;
          } else {
            const int slot = meta[c0 + i];
            if (slot >= 0 && slot < q.cap)
              ko[((size_t)(meta[256 + c0 + i] * q.nkv + (h - q.nq)) * q.cap + slot) * d + e] = r;
            else if (e == 0)
              latch_error(a.err, DEVERR_CAPACITY);
          }
        }
      } else {
        __nv_bfloat16* vo = reinterpret_cast<__nv_bfloat16*>(q.vc);
#pragma unroll 4
        for (int i = 0; i < jn; ++i) {
          const int slot = meta[c0 + i];
          if (slot >= 0 && slot < q.cap)
            vo[((size_t)(meta[256 + c0 + i] * q.nkv + (h - q.nq - q.nkv)) * q.cap + slot) * d + e] =
                __float2bfloat16_rn(staging[i * 128 + row]);
        }
      }
    }
    named_bar_sync(2, 128);
    return;
  }
  const int f = tn * 128 + row;
  if (a.epi == EPI_ADD_F32) {
    if (f < a.N) {
      // residual update: all reads first (one round trip), then the writes
      const int j0 = tt * BN + c0;
      float* o = reinterpret_cast<float*>(a.out) + (size_t)j0 * a.ldo + f;
      float old[CH];
#pragma unroll
      for (int i = 0; i < CH; ++i) old[i] = (j0 + i < a.M) ? o[(size_t)i * a.ldo] : 0.f;
#pragma unroll
      for (int i = 0; i < CH; ++i)
        if (j0 + i < a.M) o[(size_t)i * a.ldo] = old[i] + v[i];
    }
  } else if (a.epi != EPI_HEAD) {
    if (f < a.N) {
#pragma unroll
      for (int i = 0; i < CH; ++i) {
        const int j = tt * BN + c0 + i;
        if (j < a.M) {
          const size_t o = (size_t)j * a.ldo + f;
          if (a.epi == EPI_F32) reinterpret_cast<float*>(a.out)[o] = v[i];
          else reinterpret_cast<__nv_bfloat16*>(a.out)[o] = __float2bfloat16_rn(v[i]);
        }
      }
    }
  } else {
    // LM head: each warp transposes its 32 vocabulary rows x CH columns through shared
    // memory (column stride 129 floats: the column reads are free of bank conflicts) and
    // each lane reduces one column's 32 entries; the warp holding vocabulary rows 0..31
    // combines the four quarter records of its column in quarter order.
    constexpr int LDS = 129;
    const int quarter = row >> 5;
#pragma unroll
    for (int i = 0; i < CH; ++i) staging[i * LDS + row] = v[i];
    __syncwarp();
    const int j = tt * BN + c0 + lane;
    const bool live = lane < CH && j < a.M;
    const int id0 = tn * 128 + quarter * 32;
    float r[32];
    uint32_t rank_ok = 0;
    float mx = -INFINITY, se = 0.f;
    if (live) head_quarter_load(staging + lane * LDS + quarter * 32, id0, j, a.head, r, rank_ok, mx, se);
    named_bar_sync(2, 128);                  // all columns read: the staging area is free
    const int RS = 2 + 2 * a.head.K;
    float* xq = staging + lane * RS;         // quarter q's record of this column: xq + q * 32 * RS
    if (live) head_quarter_select(r, rank_ok, id0, a.head.K, mx, se, xq + quarter * 32 * RS);
    named_bar_sync(2, 128);
    if (quarter == 0 && live)
      head_quarter_merge(xq, xq + 32 * RS, xq + 64 * RS, xq + 96 * RS, a.head.K, tn, j, a.head);
    named_bar_sync(2, 128);
  }
}

// Walk over a CTA's work: the segments of its unit range [u_begin, u_end) (a segment = the
// range's piece of one weight tile), each run for token tiles 0..TT-1 in turn.
struct SegCursor {
  long long u, s0, s1, end, tile;
  int tt, TT, kb;
  __device__ __forceinline__ void init(long long ub, long long ue, int nt, int k) {
    end = ue; TT = nt; kb = k; tt = 0;
    u = s0 = ub;
    tile = ub / kb;
    s1 = min(ue, (tile + 1) * kb);
  }
  __device__ __forceinline__ bool done() const { return s0 >= end; }
  // the next unit (k-block) in issue order
  __device__ __forceinline__ void next() {
    if (++u < s1) return;
    if (++tt < TT) { u = s0; return; }
    tt = 0;
    s0 = s1;
    u = s0;
    tile = s0 / kb;
    s1 = min(end, (tile + 1) * kb);
  }
  // the start of the next (segment, token tile) item
  __device__ __forceinline__ void next_item() {
    u = s1 - 1;
    next();
  }
};

template <int BN, int MODE>
__global__ void __launch_bounds__(192, 1)
    gemm_bf16_tc(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                 const GemmArgs a) {
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
  uint64_t* fixbar = drain + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(fixbar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* bcast = reinterpret_cast<volatile int*>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = blockIdx.x, G = gridDim.x, TT = a.tiles_t;
  const long long U = a.units;
  const long long u_begin = (long long)cta * U / G, u_end = (long long)(cta + 1) * U / G;

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
    mbar_init(smem_u32(fixbar), 1);
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
      // a weight box read once is streamed past L2; with several token tiles the next ones
      // re-read it (1088 x 28672 x 4096: 294 -> 284 us)
      const uint64_t pol_w = TT > 1 ? l2_policy_evict_last() : l2_policy_evict_first();
      const uint64_t pol_x = l2_policy_evict_last();
      int stage = 0;
      uint32_t phase = 0, issued = 0, parity = 0;
      // weight tile (128 rows x 64 k); SwiGLU: 64 gate rows + the matching 64 up rows
      auto load_w = [&](uint32_t dst, const SegCursor& c, uint32_t bar) {
        const int k = (int)(c.u - c.tile * a.kb), tn = (int)c.tile;
        if constexpr (MODE == MODE_SWIGLU) {
          tma_load_2d(dst, &tmW, k * 64, tn * 64, bar, pol_w);
          tma_load_2d(dst + C::A_BYTES / 2, &tmW, k * 64, a.N + tn * 64, bar, pol_w);
        } else {
          tma_load_2d(dst, &tmW, k * 64, tn * 128, bar, pol_w);
        }
      };
      auto load_x = [&](uint32_t dst, const SegCursor& c, uint32_t bar) {
        tma_load_2d(dst, &tmX, (int)(c.u - c.tile * a.kb) * 64, c.tt * BN, bar, pol_x);
      };
      // The first ring of weight tiles does not depend on the previous kernel: issue it
      // before waiting for that kernel, then add the activation halves of those stages
      // once its outputs are visible.
      const long long steps = (u_end - u_begin) * TT;
      const int n_pre = (int)min((long long)C::STAGES, steps);
      SegCursor cur;
      cur.init(u_begin, u_end, TT, a.kb);
      {
        SegCursor c = cur;
        for (int i = 0; i < n_pre; ++i) {
          const uint32_t fb = smem_u32(full + i);
          mbar_expect_tx(fb, C::STAGE);
          load_w(smem_u32(smem + i * C::STAGE), c, fb);
          issued |= 1u << i;
          c.next();
        }
      }
      pdl_wait();
      for (int i = 0; i < n_pre; ++i) {
        load_x(smem_u32(smem + i * C::STAGE) + C::A_BYTES, cur, smem_u32(full + i));
        cur.next();
      }
      stage = n_pre % C::STAGES;
      phase = (n_pre == C::STAGES) ? 1u : 0u;
      for (long long i = n_pre; i < steps; ++i) {
        if (!mbar_wait(smem_u32(empty + stage), phase ^ 1, abort_flag, a.err)) break;
        const uint32_t fb = smem_u32(full + stage);
        mbar_expect_tx(fb, C::STAGE);
        const uint32_t sa = smem_u32(smem + stage * C::STAGE);
        load_w(sa, cur, fb);
        load_x(sa + C::A_BYTES, cur, fb);
        issued |= 1u << stage;
        parity = (parity & ~(1u << stage)) | (phase << stage);
        if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
        cur.next();
      }
      if (*abort_flag) {
        for (int s = 0; s < C::STAGES; ++s)
          if ((issued >> s) & 1) mbar_wait(smem_u32(full + s), (parity >> s) & 1, abort_flag, a.err, false);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t IDESC = idesc_bf16<BN>();
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      SegCursor c;
      c.init(u_begin, u_end, TT, a.kb);
      // one item = a segment's units for one token tile, accumulated into one TMEM buffer
      while (ok && !c.done()) {
        if (!mbar_wait(smem_u32(tempty + acc), acc_phase ^ 1, abort_flag, a.err)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * BN);
        for (long long u = c.s0; u < c.s1; ++u) {
          if (!mbar_wait(smem_u32(full + stage), phase, abort_flag, a.err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * C::STAGE);
          const uint64_t da = sdesc_sw128(sa), db = sdesc_sw128(sa + C::A_BYTES);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            tc_mma_bf16(d, da + 2 * k, db + 2 * k, IDESC, (u != c.s0 || k) ? 1u : 0u);
          tc_commit(smem_u32(empty + stage));
          if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        tc_commit(smem_u32(tfull + acc));
        acc ^= 1;
        if (!acc) acc_phase ^= 1;
        c.next_item();
      }
      if (!ok) {
        tc_commit(smem_u32(drain));
        mbar_wait(smem_u32(drain), 0, abort_flag, a.err, false);
      }
    }
  } else {
    pdl_wait();
    // epilogue chunk width (accumulator columns per TMEM load)
    constexpr int ECH = (MODE == MODE_QKV) ? 16 : C::CH;
    const int ew = warp - 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const bool leader = (ew == 0 && lane == 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    SegCursor c;
    c.init(u_begin, u_end, TT, a.kb);
    while (!c.done()) {
      const long long tile = c.tile;
      const int tn = (int)tile, tt = c.tt;
      const bool whole = (c.s0 == tile * a.kb) && (c.s1 == (tile + 1) * a.kb);
      const bool last_item = c.s1 == u_end && tt == TT - 1;   // nothing follows in the TMA ring
      const long long gtile = (long long)tn * TT + tt;        // counter index
      if (leader) bcast[0] = mbar_wait(smem_u32(tfull + acc), acc_phase, abort_flag, a.err) ? 1 : 0;
      named_bar_sync(1, 128);
      const int ok = bcast[0];
      named_bar_sync(1, 128);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
      if (whole) {
        for (int c0 = 0; c0 < BN; c0 += ECH) {
          float v[ECH];
          if constexpr (ECH == 32) tmem_ld32(tb + c0, v); else tmem_ld16(tb + c0, v);
          epi_chunk<ECH, MODE>(a, tn, tt, BN, row, c0, v, staging, ew, lane);
        }
        tc_fence_before();
        mbar_arrive(smem_u32(tempty + acc));
      } else {
        // Split tile. Its first contributor cf (whose range holds the tile's first k-block;
        // for it the tile is its last segment) owns the result; each later contributor (for
        // which the tile is its first segment) publishes a partial [BN tokens][128 features]
        // into its slot for this token tile and counts itself in. The owner waits for the
        // count, then adds the partials to its own accumulator in contributor order.
        const int cf = cta_of_unit(tile * a.kb, U, G);
        const int cl = cta_of_unit((tile + 1) * a.kb - 1, U, G);
        const int nother = cl - cf;
        constexpr uint32_t PART = (uint32_t)BN * 128 * 4;
        auto slot = [&](int q) { return a.partials + ((size_t)q * TT + tt) * BN * 128; };
        if (c.s0 != tile * a.kb) {
          float* part = slot(cta);
          for (int c0 = 0; c0 < BN; c0 += ECH) {
            float v[ECH];
            if constexpr (ECH == 32) tmem_ld32(tb + c0, v); else tmem_ld16(tb + c0, v);
#pragma unroll
            for (int i = 0; i < ECH; ++i) part[(c0 + i) * 128 + row] = v[i];
          }
          tc_fence_before();
          mbar_arrive(smem_u32(tempty + acc));
          __threadfence();
          named_bar_sync(1, 128);
          if (leader) red_release_add(reinterpret_cast<unsigned*>(a.counters + gtile), 1u);
        } else {
          // on the CTA's last item the TMA ring is idle: with room, the partials come in as
          // bulk copies, all in flight at once
          const bool bulk = last_item && (uint32_t)nother * PART <= (uint32_t)(C::STAGES * C::STAGE);
          if (leader) {
            bool ok = grid_wait(reinterpret_cast<const unsigned*>(a.counters + gtile), (unsigned)nother,
                                abort_flag, a.err, false);
            if (ok && bulk && nother > 0) {
              fence_acq_rel_gpu();
              fence_proxy_async_all();
              mbar_expect_tx(smem_u32(fixbar), (uint32_t)nother * PART);
              for (int q = 0; q < nother; ++q)
                bulk_load(smem_u32(smem + (size_t)q * PART), slot(cf + 1 + q), PART, smem_u32(fixbar));
              ok = mbar_wait(smem_u32(fixbar), 0, abort_flag, a.err);
            }
            bcast[0] = ok ? 1 : 0;
          }
          named_bar_sync(1, 128);
          if (bcast[0]) {
            if (!bulk) __threadfence();
            const float* sp = reinterpret_cast<const float*>(smem);
            for (int c0 = 0; c0 < BN; c0 += ECH) {
              float v[ECH];
              if constexpr (ECH == 32) tmem_ld32(tb + c0, v); else tmem_ld16(tb + c0, v);
              if (bulk) {
                for (int q = 0; q < nother; ++q)
#pragma unroll
                  for (int i = 0; i < ECH; ++i) v[i] += sp[(size_t)q * BN * 128 + (c0 + i) * 128 + row];
              } else {
                // two contributors' loads in flight together
                for (int cc = cf + 1; cc <= cl; cc += 2) {
                  const bool two = cc + 1 <= cl;
                  const float* p0 = slot(cc) + c0 * 128 + row;
                  const float* p1 = slot(two ? cc + 1 : cc) + c0 * 128 + row;
                  float x0[ECH], x1[ECH];
#pragma unroll
                  for (int i = 0; i < ECH; ++i) {
                    x0[i] = __ldcg(p0 + i * 128);
                    x1[i] = two ? __ldcg(p1 + i * 128) : 0.f;
                  }
#pragma unroll
                  for (int i = 0; i < ECH; ++i) v[i] += x0[i];
                  if (two) {
#pragma unroll
                    for (int i = 0; i < ECH; ++i) v[i] += x1[i];
                  }
                }
              }
              epi_chunk<ECH, MODE>(a, tn, tt, BN, row, c0, v, staging, ew, lane);
            }
          }
          tc_fence_before();
          mbar_arrive(smem_u32(tempty + acc));
          if (leader) a.counters[gtile] = 0;
        }
        named_bar_sync(1, 128);
      }
      acc ^= 1;
      if (!acc) acc_phase ^= 1;
      c.next_item();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// ---- whole-tile schedule for several token tiles ----------------------------------------------
// Items are (weight tile, token tile) pairs, tile-major (the token tiles of a weight tile
// follow one another, so they re-read its boxes from L2); CTA c takes items
// [c * I / G, (c + 1) * I / G). Each item's k-range is cut where the stream-K schedule of the
// same (N, K) cuts that weight tile (unit ranges [c * U / Gs, (c + 1) * U / Gs) of Gs CTAs),
// every piece is accumulated into its own TMEM buffer (accumulate flag cleared at its first
// k-block; two buffers, so the next piece's MMAs run while the epilogue reads this one) and
// the epilogue adds the pieces in k order in fp32 into a third TMEM buffer - the additions
// the stream-K owner makes with its contributors' partials - so the outputs have the
// stream-K schedule's bits, with no partials and no waits between CTAs.
struct PieceCursor {
  long long item, end, U;
  int TT, kb, Gs;
  int tile, tt, cf, cl, p;
  long long k0, k1;        // the current piece's units [k0, k1)
  __device__ __forceinline__ void init(long long b, long long e, int TT_, int kb_, long long U_, int Gs_) {
    item = b; end = e; TT = TT_; kb = kb_; U = U_; Gs = Gs_;
    if (item < end) set_item();
  }
  __device__ __forceinline__ void set_item() {
    tile = (int)(item / TT);
    tt = (int)(item - (long long)tile * TT);
    cf = cta_of_unit((long long)tile * kb, U, Gs);
    cl = cta_of_unit((long long)(tile + 1) * kb - 1, U, Gs);
    p = 0;
    set_piece();
  }
  __device__ __forceinline__ void set_piece() {
    k0 = max((long long)tile * kb, (long long)(cf + p) * U / Gs);
    k1 = min((long long)(tile + 1) * kb, (long long)(cf + p + 1) * U / Gs);
  }
  __device__ __forceinline__ bool done() const { return item >= end; }
  __device__ __forceinline__ bool last_piece() const { return cf + p == cl; }
  __device__ __forceinline__ void next() {
    if (cf + p < cl) { ++p; set_piece(); return; }
    if (++item < end) set_item();
  }
};

template <int BN, int MODE>
__global__ void __launch_bounds__(192, 1)
    gemm_bf16_tc_whole(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                       const GemmArgs a, int Gs) {
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
  const int cta = blockIdx.x, G = gridDim.x, TT = a.tiles_t, kb = a.kb;
  const long long I = a.units / kb * TT;
  const long long i_begin = (long long)cta * I / G, i_end = (long long)(cta + 1) * I / G;

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
  constexpr uint32_t WCOLS = 3 * BN <= 256 ? 256 : 512;   // two piece buffers and the sum
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), WCOLS);
  pdl_trigger();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol_w = l2_policy_evict_last();   // the next token tiles re-read it
      const uint64_t pol_x = l2_policy_evict_last();
      int stage = 0;
      uint32_t phase = 0, issued = 0, parity = 0;
      auto load_w = [&](uint32_t dst, int tile, int k, uint32_t bar) {
        if constexpr (MODE == MODE_SWIGLU) {
          tma_load_2d(dst, &tmW, k * 64, tile * 64, bar, pol_w);
          tma_load_2d(dst + C::A_BYTES / 2, &tmW, k * 64, a.N + tile * 64, bar, pol_w);
        } else {
          tma_load_2d(dst, &tmW, k * 64, tile * 128, bar, pol_w);
        }
      };
      auto load_x = [&](uint32_t dst, int tt, int k, uint32_t bar) {
        tma_load_2d(dst, &tmX, k * 64, tt * BN, bar, pol_x);
      };
      // (item, k-block) steps in issue order
      const long long steps = (i_end - i_begin) * kb;
      const int n_pre = (int)min((long long)C::STAGES, steps);
      // the first ring of weight boxes does not depend on the previous kernel
      for (int i = 0; i < n_pre; ++i) {
        const long long it = i_begin + i / kb;
        const uint32_t fb = smem_u32(full + i);
        mbar_expect_tx(fb, C::STAGE);
        load_w(smem_u32(smem + i * C::STAGE), (int)(it / TT), i % kb, fb);
        issued |= 1u << i;
      }
      pdl_wait();
      for (int i = 0; i < n_pre; ++i) {
        const long long it = i_begin + i / kb;
        load_x(smem_u32(smem + i * C::STAGE) + C::A_BYTES, (int)(it % TT), i % kb, smem_u32(full + i));
      }
      stage = n_pre % C::STAGES;
      phase = (n_pre == C::STAGES) ? 1u : 0u;
      long long it = i_begin + n_pre / kb;
      int k = n_pre % kb;
      for (long long i = n_pre; i < steps; ++i) {
        if (!mbar_wait(smem_u32(empty + stage), phase ^ 1, abort_flag, a.err)) break;
        const uint32_t fb = smem_u32(full + stage);
        mbar_expect_tx(fb, C::STAGE);
        const uint32_t sa = smem_u32(smem + stage * C::STAGE);
        load_w(sa, (int)(it / TT), k, fb);
        load_x(sa + C::A_BYTES, (int)(it % TT), k, fb);
        issued |= 1u << stage;
        parity = (parity & ~(1u << stage)) | (phase << stage);
        if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
        if (++k == kb) { k = 0; ++it; }
      }
      if (*abort_flag) {
        for (int s = 0; s < C::STAGES; ++s)
          if ((issued >> s) & 1) mbar_wait(smem_u32(full + s), (parity >> s) & 1, abort_flag, a.err, false);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t IDESC = idesc_bf16<BN>();
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      PieceCursor c;
      c.init(i_begin, i_end, TT, kb, a.units, Gs);
      while (ok && !c.done()) {
        if (!mbar_wait(smem_u32(tempty + acc), acc_phase ^ 1, abort_flag, a.err)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * BN);
        for (long long u = c.k0; u < c.k1; ++u) {
          if (!mbar_wait(smem_u32(full + stage), phase, abort_flag, a.err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * C::STAGE);
          const uint64_t da = sdesc_sw128(sa), db = sdesc_sw128(sa + C::A_BYTES);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma_bf16(d, da + 2 * kk, db + 2 * kk, IDESC, (u != c.k0 || kk) ? 1u : 0u);
          tc_commit(smem_u32(empty + stage));
          if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        tc_commit(smem_u32(tfull + acc));
        acc ^= 1;
        if (!acc) acc_phase ^= 1;
        c.next();
      }
      if (!ok) {
        tc_commit(smem_u32(drain));
        mbar_wait(smem_u32(drain), 0, abort_flag, a.err, false);
      }
    }
  } else {
    pdl_wait();
    constexpr int ECH = (MODE == MODE_QKV) ? 16 : C::CH;
    const int ew = warp - 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const bool leader = (ew == 0 && lane == 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    const uint32_t lane_base = tmem_base + ((uint32_t)(quarter * 32) << 16);
    const uint32_t ts = lane_base + (uint32_t)(2 * BN);   // the running sum
    PieceCursor c;
    c.init(i_begin, i_end, TT, kb, a.units, Gs);
    while (!c.done()) {
      if (leader) bcast[0] = mbar_wait(smem_u32(tfull + acc), acc_phase, abort_flag, a.err) ? 1 : 0;
      named_bar_sync(1, 128);
      const int ok = bcast[0];
      named_bar_sync(1, 128);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tb = lane_base + (uint32_t)(acc * BN);
      const bool first = c.p == 0, last = c.last_piece();
      if (last && !first) {
        // the last piece: sum + piece, then the epilogue; the buffer is free once read
        for (int c0 = 0; c0 < BN; c0 += ECH) {
          float v[ECH], w[ECH];
          if constexpr (ECH == 32) { tmem_ld32(tb + c0, v); tmem_ld32(ts + c0, w); }
          else { tmem_ld16(tb + c0, v); tmem_ld16(ts + c0, w); }
#pragma unroll
          for (int i = 0; i < ECH; ++i) v[i] = w[i] + v[i];
          if (c0 + ECH >= BN) {
            tc_fence_before();
            mbar_arrive(smem_u32(tempty + acc));
          }
          epi_chunk<ECH, MODE>(a, c.tile, c.tt, BN, row, c0, v, staging, ew, lane);
        }
      } else if (last) {
        for (int c0 = 0; c0 < BN; c0 += ECH) {
          float v[ECH];
          if constexpr (ECH == 32) tmem_ld32(tb + c0, v); else tmem_ld16(tb + c0, v);
          if (c0 + ECH >= BN) {
            tc_fence_before();
            mbar_arrive(smem_u32(tempty + acc));
          }
          epi_chunk<ECH, MODE>(a, c.tile, c.tt, BN, row, c0, v, staging, ew, lane);
        }
      } else {
        // a piece before the last: into the running sum
        for (int c0 = 0; c0 < BN; c0 += 16) {
          float v[16], w[16];
          tmem_ld16(tb + c0, v);
          if (!first) {
            tmem_ld16(ts + c0, w);
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = w[i] + v[i];
          }
          tmem_st16(ts + c0, v);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(smem_u32(tempty + acc));
      }
      acc ^= 1;
      if (!acc) acc_phase ^= 1;
      c.next();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, WCOLS);
  }
}

// ---- host side ----------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// bf16 row-major [rows][K] matrix (row stride ld, 0 = K), boxes of 64 (K) x box_rows,
// 128-byte swizzle.
static bool make_map(CUtensorMap* m, const void* ptr, long long rows, long long K, int box_rows,
                     bool use_cache = true, long long ld = 0) {
  if (ld <= 0) ld = K;
  static std::map<std::tuple<const void*, long long, long long, int, long long>, CUtensorMap> cache;
  static std::mutex mu;
  auto key = std::make_tuple(ptr, rows, K, box_rows, ld);
  if (use_cache) {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) { *m = it->second; return true; }
  }
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  if (!use_cache) return true;
  std::lock_guard<std::mutex> lock(mu);
  if (cache.size() > 4096) cache.clear();
  cache[key] = *m;
  return true;
}

bool make_tmap_bf16(CUtensorMap* m, const void* ptr, long long rows, long long K, int box_rows, long long ld) {
  return make_map(m, ptr, rows, K, box_rows, true, ld);
}

// Host caches kept per device: a process may drive several GPUs, each with its own SM
// count and its own per-function attributes.
constexpr int kMaxDevices = 64;

int device_sm_count() {
  static std::mutex mu;
  static int n[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
  std::lock_guard<std::mutex> lock(mu);
  if (!n[dev]) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 1;
    n[dev] = v;
  }
  return n[dev];
}

cudaError_t raise_smem_limit(const void* func, int bytes) {
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, int> limit;   // the limit last set, per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_pair(dev, func);
  auto it = limit.find(key);
  if (it != limit.end() && it->second >= bytes) return cudaSuccess;   // only ever raised
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) limit[key] = bytes;
  return e;
}

static int num_sms() { return device_sm_count(); }

// EAGLE_GEMM_WHOLE=0 keeps the stream-K schedule for every row count (same results).
static bool whole_tiles_enabled() {
  static const bool on = !(getenv("EAGLE_GEMM_WHOLE") && strcmp(getenv("EAGLE_GEMM_WHOLE"), "0") == 0);
  return on;
}

int gemm_bn_for(int M) {
  if (M <= 16) return 16;
  if (M <= 32) return 32;
  if (M <= 64) return 64;
  if (M <= 128) return 128;
  return 256;
}

// Split-tile partial sums: one slot of BN x 128 floats per (CTA, token tile).
size_t gemm_bf16_scratch_bytes(int max_rows) {
  const size_t tt = max_rows > 256 ? (size_t)(max_rows + 255) / 256 : 1;
  return (size_t)num_sms_cap() * tt * 256 * 128 * sizeof(float);
}

template <int BN, int MODE>
static cudaError_t launch_bn(const CUtensorMap& mw, const CUtensorMap& mx, GemmArgs& a, int G, cudaStream_t st) {
  using C = TcCfg<BN>;
  cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(gemm_bf16_tc<BN, MODE>), C::SMEM);
  if (e != cudaSuccess) return e;
  launch_k(gemm_bf16_tc<BN, MODE>, G, 192, C::SMEM, st, mw, mx, a);
  return cudaGetLastError();
}

template <int MODE>
static cudaError_t launch_whole(const CUtensorMap& mw, const CUtensorMap& mx, GemmArgs& a, int G, int Gs,
                                cudaStream_t st) {
  using C = TcCfg<128>;
  cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(gemm_bf16_tc_whole<128, MODE>), C::SMEM);
  if (e != cudaSuccess) return e;
  launch_k(gemm_bf16_tc_whole<128, MODE>, G, 192, C::SMEM, st, mw, mx, a, Gs);
  return cudaGetLastError();
}

template <int BN>
static cudaError_t launch_mode(const CUtensorMap& mw, const CUtensorMap& mx, GemmArgs& a, int G, cudaStream_t st) {
  if (a.epi == EPI_SWIGLU || a.epi == EPI_GU) return launch_bn<BN, MODE_SWIGLU>(mw, mx, a, G, st);
  if (a.epi == EPI_QKV) return launch_bn<BN, MODE_QKV>(mw, mx, a, G, st);
  return launch_bn<BN, MODE_GENERIC>(mw, mx, a, G, st);
}

int gemm_bf16(cudaStream_t st, const void* W, int N, int K, const void* X, int M, int epi, void* out,
              int ldo, float* partials, size_t partial_floats, int* counters, int counters_len, int* err,
              const HeadParams* head, bool cache_maps, const QkvEpi* qkv) {
  if (M <= 0 || N <= 0 || K <= 0 || (K % 8) != 0 || !W || !X) return -1;
  if ((reinterpret_cast<uintptr_t>(W) | reinterpret_cast<uintptr_t>(X)) & 15) return -1;
  const bool paired = epi == EPI_SWIGLU || epi == EPI_GU;
  if (paired && N % 64) return -1;
  if (epi == EPI_QKV && (!qkv || qkv->d < 2 || qkv->d % 2 || 128 % qkv->d || N != (qkv->nq + 2 * qkv->nkv) * qkv->d))
    return -1;
  const int tiles_n = paired ? N / 64 : (N + 127) / 128;
  const int kb = (K + 63) / 64;
  const long long units = (long long)tiles_n * kb;
  // the stream-K ranges depend on (N, K, SM count) only
  int G = std::min(num_sms(), num_sms_cap());
  if (G > units) G = (int)units;
  // More than one 128-token tile and fewer weight tiles than CTAs (every tile split across
  // CTAs, whose fixups then serialise per token tile): whole (weight tile, token tile) items
  // cut at the same k-points, so the same bits (measured at 1088 tokens: QKV 155 -> 66 us,
  // O 178 -> 47, down 238 -> 142; with more tiles than CTAs, gate/up and the LM head, the
  // stream-K schedule with 256-token tiles stays faster)
  const bool whole = M > 128 && tiles_n < G && epi != EPI_HEAD && whole_tiles_enabled();
  const int BN = whole ? 128 : gemm_bn_for(M);
  const int tiles_t = (M + BN - 1) / BN;
  if (!whole && (long long)tiles_n * tiles_t > counters_len) return -2;
  if (!whole && (size_t)G * tiles_t * BN * 128 > partial_floats) return -2;
  CUtensorMap mw, mx;
  if (paired) {
    if (!make_map(&mw, W, 2LL * N, K, 64, cache_maps)) return -3;
  } else if (!make_map(&mw, W, N, K, 128, cache_maps)) {
    return -3;
  }
  if (!make_map(&mx, X, M, K, BN, cache_maps)) return -3;
  GemmArgs a{};
  a.M = M; a.N = N; a.K = K; a.epi = epi; a.out = out; a.ldo = ldo;
  a.tiles_t = tiles_t; a.kb = kb; a.units = units;
  a.partials = partials; a.counters = counters; a.err = err;
  if (head) a.head = *head;
  if (qkv) a.qkv = *qkv;
  cudaError_t e;
  if (whole) {
    const int Gw = (int)std::min<long long>(std::min(num_sms(), num_sms_cap()), (long long)tiles_n * tiles_t);
    if (paired) e = launch_whole<MODE_SWIGLU>(mw, mx, a, Gw, G, st);
    else if (epi == EPI_QKV) e = launch_whole<MODE_QKV>(mw, mx, a, Gw, G, st);
    else e = launch_whole<MODE_GENERIC>(mw, mx, a, Gw, G, st);
    return e == cudaSuccess ? 0 : -4;
  }
  switch (BN) {
    case 16: e = launch_mode<16>(mw, mx, a, G, st); break;
    case 32: e = launch_mode<32>(mw, mx, a, G, st); break;
    case 64: e = launch_mode<64>(mw, mx, a, G, st); break;
    case 128: e = launch_mode<128>(mw, mx, a, G, st); break;
    default: e = launch_mode<256>(mw, mx, a, G, st); break;
  }
  return e == cudaSuccess ? 0 : -4;
}

}  // namespace eagle
