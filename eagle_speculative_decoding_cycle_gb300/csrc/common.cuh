// Shared device helpers for the EAGLE cycle kernels (sm_103a).
//
// Contents: bf16/f32 storage traits, warp reductions, a device status word that
// kernels latch errors into instead of trapping, bounded mbarrier waits, TMA and
// tcgen05 inline-PTX wrappers, and the Philox4x32-10 generator.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#define EAGLE_DEV __device__ __forceinline__

// ---- device error codes latched into the context's status word -------------------------
enum : int {
  DEVERR_NONE = 0,
  DEVERR_MBAR_TIMEOUT = 1,    // an mbarrier wait exceeded its time limit
  DEVERR_BOUNDS = 2,          // an index (token, slot, node) was out of range
  DEVERR_CAPACITY = 3,        // a sequence outgrew its KV capacity
};

// A wait that has not completed within this many nanoseconds is abandoned.
#define EAGLE_WAIT_LIMIT_NS 2000000000ull

// Programmatic dependent launch: every kernel waits for its predecessor grid (and so,
// transitively, for all earlier ones) before reading their outputs or writing anything,
// then lets its own dependents start launching. Triggering only after the wait bounds the
// look-ahead to one kernel: when a kernel's pre-wait prologue runs, every grid but its
// immediate predecessor has finished, which the attention's early reads of context keys rely
// on (triggering first let whole chains of kernels launch ahead and broke them). Both are
// no-ops for a launch without the programmatic-serialization attribute.
EAGLE_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
EAGLE_DEV void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
#define PDL_ENTRY() \
  do {              \
    pdl_wait();     \
    pdl_trigger();  \
  } while (0)

EAGLE_DEV void latch_error(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// ---- shared element-wise arithmetic (one definition, so fused and separate kernels agree
// bit for bit) --------------------------------------------------------------------------------
// Rotate-half RoPE of the pair (a = x[i], b = x[i + d/2]) by the angle with cosine c, sine s.
__device__ __forceinline__ void rope_pair(float a, float b, float c, float s, float& lo, float& hi) {
  lo = __fsub_rn(__fmul_rn(a, c), __fmul_rn(b, s));
  hi = __fadd_rn(__fmul_rn(b, c), __fmul_rn(a, s));
}
// SwiGLU gate: silu(g) * u.
__device__ __forceinline__ float silu_mul(float g, float u) { return __fmul_rn(__fdiv_rn(g, __fadd_rn(1.f, expf(-g))), u); }
// bf16 paths (row kernel, GEMM epilogue): the same product with the fast
// exponential and divide; their relative error (~1e-6) is far below bf16 rounding. For
// g < -87 the denominator overflows and the result is 0, the limit of silu.
__device__ __forceinline__ float silu_mul_bf16(float g, float u) {
  return __fmul_rn(__fdividef(g, __fadd_rn(1.f, __expf(-g))), u);
}

// ---- element traits ---------------------------------------------------------------------
template <typename T> struct Elem;
template <> struct Elem<float> {
  static EAGLE_DEV float load(const float* p) { return *p; }
  static EAGLE_DEV float to_f(float v) { return v; }
  static EAGLE_DEV float from_f(float v) { return v; }
};
template <> struct Elem<__nv_bfloat16> {
  static EAGLE_DEV float load(const __nv_bfloat16* p) { return __bfloat162float(*p); }
  static EAGLE_DEV float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
  static EAGLE_DEV __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
};

EAGLE_DEV float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
EAGLE_DEV float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Monotonic map of a float onto uint32 (larger float -> larger key).
EAGLE_DEV uint32_t f32_order_key(float f) {
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// "a ranks before b": larger value first, then lower id.
EAGLE_DEV bool rank_before(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// Order-preserving 32-bit key of a float (larger value, larger key; -0 and +0 map to one
// key) and its inverse, so that a warp takes a maximum with one redux.sync instead of a
// shuffle butterfly.
EAGLE_DEV uint32_t f2key(float v) {
  const uint32_t b = __float_as_uint(v + 0.f);   // -0 -> +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
EAGLE_DEV float key2f(uint32_t k) { return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k); }

// The warp's best (value, id) of one candidate per lane in the rank_before order: the
// largest value, then the smallest id among the lanes that hold it. Empty lanes carry
// (-inf, 0x7fffffff).
EAGLE_DEV void warp_best(float v, int id, float& bv, int& bi) {
  const uint32_t kv = f2key(v);
  const uint32_t kmax = __reduce_max_sync(0xffffffffu, kv);
  bi = (int)__reduce_min_sync(0xffffffffu, kv == kmax ? (uint32_t)id : 0xffffffffu);
  bv = key2f(kmax);
}

// ---- Philox4x32-10 (Salmon et al., SC'11) ---------------------------------------------------
struct u32x4 { uint32_t x, y, z, w; };

EAGLE_DEV u32x4 philox4x32_10(u32x4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) { k0 += 0x9E3779B9u; k1 += 0xBB67AE85u; }
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = u32x4{hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0};
  }
  return c;
}

// Uniform strictly inside (0,1), exact in fp32: ((x >> 9) + 0.5) * 2^-23.
EAGLE_DEV float philox_uniform(uint32_t x) {
  return (float)((x >> 9) * 2u + 1u) * 5.9604644775390625e-08f;   // (2q+1) * 2^-24
}

enum : uint32_t { STREAM_PLANT = 2, STREAM_ACCEPT = 3, STREAM_GUMBEL = 4, STREAM_PLAIN = 5 };
#define PREFILL_CYCLE 0xFFFFFFFFu

// One uniform keyed by (seed; counter = (a, b, cycle, seq << 8 | stream)), word 0.
EAGLE_DEV float draw_uniform(uint64_t seed, uint32_t stream, uint32_t seq, uint32_t cycle,
                             uint32_t a, uint32_t b) {
  u32x4 o = philox4x32_10(u32x4{a, b, cycle, (seq << 8) | stream}, (uint32_t)seed,
                          (uint32_t)(seed >> 32));
  return philox_uniform(o.x);
}

// ---- mbarrier / TMA / tcgen05 wrappers ------------------------------------------------------
EAGLE_DEV uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

EAGLE_DEV uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

EAGLE_DEV void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

EAGLE_DEV void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

EAGLE_DEV bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait. Returns false when the wait gave up: either the CTA's abort flag was
// already raised by another role, or the time limit passed (then the flag and the
// device status word are set). `honor_abort` = false is used while draining.
EAGLE_DEV bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* err,
                         bool honor_abort = true) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    if (mbar_try(bar, parity)) return true;
    if (honor_abort && *abort_flag) return false;
    if (globaltimer() - t0 > EAGLE_WAIT_LIMIT_NS) {
      *abort_flag = 1;
      latch_error(err, DEVERR_MBAR_TIMEOUT);
      return false;
    }
  }
}

EAGLE_DEV void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

EAGLE_DEV void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// 2D tiled TMA load into shared memory, completion signalled on `bar` (complete_tx).
EAGLE_DEV void tma_load_2d(uint32_t dst, const void* tmap, int c0, int c1, uint32_t bar,
                           uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(c0), "r"(c1), "l"(policy)
      : "memory");
}

// Orders this thread's earlier generic-proxy memory accesses with its later async-proxy
// ones (bulk / tensor copies).
EAGLE_DEV void fence_proxy_async_all() { asm volatile("fence.proxy.async;" ::: "memory"); }

// Contiguous bulk copy global -> shared memory (16-byte aligned addresses and size),
// completion signalled on `bar` (complete_tx).
EAGLE_DEV void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
               : "memory");
}

// Bring one 2D tile of a tensor into L2 without touching shared memory.
EAGLE_DEV void tma_prefetch_l2_2d(const void* tmap, int c0, int c1) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(tmap)),
               "r"(c0), "r"(c1)
               : "memory");
}

EAGLE_DEV uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
EAGLE_DEV uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

EAGLE_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
EAGLE_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Issued by one full warp.
EAGLE_DEV void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
EAGLE_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, kind::f16 (bf16 inputs, fp32 accumulate).
EAGLE_DEV void tc_mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05.mma issued so far by this thread has completed.
EAGLE_DEV void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

// 32 lanes x 32 consecutive fp32 columns; thread i receives lane (base + i).
EAGLE_DEV void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

EAGLE_DEV void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Stores of 32 lanes x 16 consecutive fp32 columns (thread i writes lane base + i); the
// caller waits with tmem_wait_st before reading them back.
EAGLE_DEV void tmem_st16(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
      ::"r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15]))
      : "memory");
}
EAGLE_DEV void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

EAGLE_DEV void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}
