// Pieces of the tcgen05 weight-streaming GEMM: stage geometry, the shared-memory operand descriptor, and the stream-K split.
#pragma once

#include "common.cuh"

namespace eagle {

// Stage = one 128-row x 64-k weight box (A) + one BN-row x 64-k activation box (B), both
// bf16 with the 128-byte swizzle. The ring fills ~192 KB; TMEM holds two BN-column fp32
// accumulators so one tile's epilogue overlaps the next tile's main loop.
template <int BN>
struct TcCfg {
  static constexpr int A_BYTES = 128 * 64 * 2;
  static constexpr int B_BYTES = BN * 64 * 2;
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int STAGES = (196608 / STAGE) > 12 ? 12 : (196608 / STAGE);
  static constexpr int TMEM_COLS = (2 * BN < 32) ? 32 : 2 * BN;
  static constexpr int CH = BN < 32 ? BN : 32;
  static constexpr int STAGING = 32 * 128 * 4 + 3 * 256 * 4;   // epilogue values + per-column metadata
  static constexpr int SMEM = 1024 + STAGES * STAGE + STAGING + 512;
};

// K-major operand tile, rows of 64 bf16 (128 bytes) with the 128-byte swizzle, 8-row
// atoms 1024 bytes apart. Start address, stride byte offset 1024, descriptor version 1,
// layout SWIZZLE_128B.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFF) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// kind::f16 instruction descriptor: bf16 A and B, fp32 accumulate, both K-major,
// N = BN, M = 128.
template <int BN>
__device__ __forceinline__ constexpr uint32_t idesc_bf16() {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

// Stream-K: units [c * U / G, (c + 1) * U / G) belong to CTA c; the CTA owning unit u.
__device__ __forceinline__ int cta_of_unit(long long u, long long U, int G) {
  return (int)(((u + 1) * G - 1) / U);
}

EAGLE_DEV void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
EAGLE_DEV void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

EAGLE_DEV unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

EAGLE_DEV bool err_raised(const int* err) { return *reinterpret_cast<const volatile int*>(err) != 0; }

// Bounded wait until *bar >= target. Gives up (false) on the CTA's abort flag, on an error
// latched by another CTA when `watch_err` is set, or after the time limit (then latches a
// timeout).
EAGLE_DEV bool grid_wait(const unsigned* bar, unsigned target, volatile int* abort_flag, int* err,
                         bool watch_err = true) {
  if (ld_acquire_u32(bar) >= target) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t spins = 1;; ++spins) {
    if (ld_acquire_u32(bar) >= target) return true;
    if (*abort_flag || (watch_err && (spins & 255u) == 0 && err_raised(err))) { *abort_flag = 1; return false; }
    if (globaltimer() - t0 > EAGLE_WAIT_LIMIT_NS) {
      *abort_flag = 1;
      latch_error(err, DEVERR_MBAR_TIMEOUT);
      return false;
    }
  }
}

}  // namespace eagle
