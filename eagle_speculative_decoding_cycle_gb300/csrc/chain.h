// Layer chain program (see chain.cu): the host describes a short sequence of dependent
// steps -- tensor-core projections and row ops -- that one persistent launch executes.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace eagle {

enum : int { CH_GEMM = 0, CH_RMSNORM = 1, CH_SWIGLU = 2, CH_ROPE = 3, CH_CONVERT = 4, CH_EMBED = 5, CH_CONCAT = 6 };
constexpr int CHAIN_MAX_STEPS = 16;
constexpr int CHAIN_MAX_GEMMS = 4;

// One step over the program's M rows (all activations bf16 unless stated).
//  CH_GEMM     out[M][ldo] (epi EPI_F32 / EPI_BF16 / EPI_ADD_F32) = X[M][K] W[N][K]^T
//  CH_RMSNORM  out[r][0:H] (row stride ldo) = in[r] * rsqrt(mean(in[r]^2) + eps) * aux,
//              in fp32 (in_bf16 = 0) or bf16, row stride ldi
//  CH_SWIGLU   out[M][H] = silu(in[r][i]) * in[r][H + i], in fp32 [M][2H]
//  CH_ROPE     the rotary embedding and KV-cache write described by ChainArgs::rope
//  CH_CONVERT  out[r][0:H] (row stride ldo) = in fp32 [r][0:H] (row stride ldi)
//  CH_EMBED    out fp32 [M][H] = aux[idx[r]] (table of V rows)
//  CH_CONCAT   out [M][2H] = [aux[idx[r]] ; in[idx2[r]]] (table of V rows; in [*][H])
//
// A GEMM step splits its (tile, k-block) units stream-K over the CTAs; the last contributor
// to a split tile (per-tile ticket) sums the partial tiles in contributor order and writes
// the tile, so every step's output is complete when the CTAs pass its barrier.
struct ChainStep {
  int kind;
  int gemm;               // filled by chain_run: tensor-map pair index
  int N, K, epi, ldo;
  int tiles_t, kb;        // filled by chain_run
  long long units;        // filled by chain_run
  void* out;
  const void* in;
  int ldi, in_bf16, H, V;
  const void* aux;
  const int* idx;
  const int* idx2;
  float eps;
};

struct ChainRope {
  const float* qkv;       // [M][(nq + 2 nkv) d] fp32
  int nq, nkv, d, cap;
  const int* pos;
  const int* slot;
  const int* seq;
  const float* cos;       // [positions][d / 2]
  const float* sin;
  void* q;                // [M][nq][d]
  void* kc;               // [(seq * nkv + h) * cap + slot][d]
  void* vc;
};

struct ChainArgs {
  int nsteps, M;
  ChainStep s[CHAIN_MAX_STEPS];
  ChainRope rope;
  float* partials;        // stream-K partial tiles, 2 per CTA
  int* counters;          // per-tile arrival tickets, zero between launches
  unsigned* bar;          // [2] barrier arrivals and exit tickets, zero between launches
  int* err;
};

struct ChainMaps {
  CUtensorMap w[CHAIN_MAX_GEMMS];
  CUtensorMap x[CHAIN_MAX_GEMMS];
};

struct ChainGemm {
  const void* W;          // [N][K] bf16
  const void* X;          // [M][ldx] bf16
  long long ldx;          // 0 = K
};

struct ChainProgram {
  int nsteps = 0, M = 0;
  ChainArgs args{};
  ChainGemm gemm[CHAIN_MAX_STEPS]{};
  float* partials = nullptr;
  int* counters = nullptr;
  int counters_len = 0;
  unsigned* bar = nullptr;
  int* err = nullptr;

  ChainStep& add(int kind) {
    ChainStep& s = args.s[nsteps++];
    s = ChainStep{};
    s.kind = kind;
    return s;
  }
  void add_gemm(const void* W, int N, int K, const void* X, int epi, void* out, int ldo) {
    gemm[nsteps] = ChainGemm{W, X, 0};
    ChainStep& s = add(CH_GEMM);
    s.N = N; s.K = K; s.epi = epi; s.out = out; s.ldo = ldo;
  }
};

// Returns 0, or -1 (bad program), -2 (too many units), -3 (tensor map), -4 (launch).
int chain_run(cudaStream_t st, const ChainProgram& p);

}  // namespace eagle
