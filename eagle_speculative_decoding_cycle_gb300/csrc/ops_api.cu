// Kernel-level C ABI (eagle_ops.h): each entry point runs one of the cycle's kernels on
// caller-provided device buffers.
#include <cmath>
#include <cstring>

#include "../../include/eagle.h"
#include "../../include/eagle_ops.h"
#include "common.cuh"
#include "cycle.h"
#include "kernels.h"
#include "lmhead.cuh"

using namespace eagle;

namespace {
size_t al(size_t x) { return (x + 255) / 256 * 256; }
int tiles_for(int M, int N) {
  const int BN = gemm_bn_for(M);
  return ((N + 127) / 128) * ((M + BN - 1) / BN);
}
}  // namespace

extern "C" {

size_t eagle_op_gemm_scratch_bytes(int M, int N) {
  if (M <= 0 || N <= 0) return 0;
  return al(gemm_bf16_scratch_bytes(M)) + al((size_t)tiles_for(M, N) * sizeof(int));
}

int eagle_op_gemm(int dtype, void* stream, const void* W, int N, int K, const void* X, int M, int epi, void* out,
                  int ldo, void* scratch, size_t scratch_bytes) {
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (!W || !X || !out || M <= 0 || N <= 0 || K <= 0 || ldo < N) return EAGLE_EINVAL;
  if (dtype == EAGLE_DTYPE_F32) {
    if (epi != EPI_F32 && epi != EPI_ADD_F32) return EAGLE_EINVAL;
    return gemm_f32(st, (const float*)W, N, K, (const float*)X, M, epi, (float*)out, ldo) == 0 ? EAGLE_OK : EAGLE_ECUDA;
  }
  if (dtype != EAGLE_DTYPE_BF16 || epi < 0 || epi == EPI_HEAD || epi > EPI_SWIGLU || K % 8) return EAGLE_EINVAL;
  const int tiles_N = epi == EPI_SWIGLU ? 2 * N : N;   // SwiGLU: W has 2N rows, tiles of 64 + 64
  if (!scratch || scratch_bytes < eagle_op_gemm_scratch_bytes(M, tiles_N)) return EAGLE_ECAPACITY;
  float* part = reinterpret_cast<float*>(scratch);
  int* cnt = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(scratch) + al(gemm_bf16_scratch_bytes(M)));
  const int r = gemm_bf16(st, W, N, K, X, M, epi, out, ldo, part, gemm_bf16_scratch_bytes(M) / sizeof(float), cnt,
                          tiles_for(M, tiles_N), nullptr, nullptr);
  return r == 0 ? EAGLE_OK : (r == -4 ? EAGLE_ECUDA : EAGLE_EINVAL);
}

size_t eagle_op_lm_head_scratch_bytes(int dtype, int V, int M, int K) {
  if (V <= 0 || M <= 0 || K < 1 || K > 16) return 0;
  size_t s = al(head_part_bytes(V, M, K));
  if (dtype == EAGLE_DTYPE_F32) s += al((size_t)M * V * sizeof(float));
  else s += eagle_op_gemm_scratch_bytes(M, V);
  return s;
}

int eagle_op_lm_head(int dtype, void* stream, const void* W_lm, int V, int H, const void* X, int M, int K, float inv_t,
                     int gumbel, int lse_excl, const int32_t* specials, int S, float* spec_logit,
                     const int32_t* row_seq, const int32_t* row_key, uint32_t cycle, uint64_t seed, int stream_id,
                     int32_t* top_id, float* top_val, float* lse, void* scratch, size_t scratch_bytes) {
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (!W_lm || !X || !top_id || !top_val || !lse || V <= 0 || H <= 0 || M <= 0 || K < 1 || K > 16) return EAGLE_EINVAL;
  if (specials && (S < 1 || !spec_logit)) return EAGLE_EINVAL;
  if (!scratch || scratch_bytes < eagle_op_lm_head_scratch_bytes(dtype, V, M, K)) return EAGLE_ECAPACITY;
  HeadParams p{};
  p.vocab = V; p.n_rows = M; p.K = K; p.inv_t = inv_t; p.gumbel = gumbel; p.lse_excl = lse_excl;
  p.specials = specials; p.S = specials ? S : 0; p.spec_logit = spec_logit;
  p.row_seq = row_seq; p.row_key = row_key; p.cycle_const = cycle; p.stream = (uint32_t)stream_id; p.seed = seed;
  uint8_t* s = reinterpret_cast<uint8_t*>(scratch);
  p.part = reinterpret_cast<float*>(s);
  s += al(head_part_bytes(V, M, K));
  p.n_tiles = (V + 127) / 128;
  p.top_id = top_id; p.top_val = top_val; p.lse = lse;
  if (dtype == EAGLE_DTYPE_F32) {
    float* logits = reinterpret_cast<float*>(s);
    if (gemm_f32(st, (const float*)W_lm, V, H, (const float*)X, M, EPI_F32, logits, V)) return EAGLE_ECUDA;
    if (head_partials_from_logits(st, logits, V, p)) return EAGLE_ECUDA;
  } else if (dtype == EAGLE_DTYPE_BF16) {
    if (H % 8) return EAGLE_EINVAL;
    float* part = reinterpret_cast<float*>(s);
    int* cnt = reinterpret_cast<int*>(s + al(gemm_bf16_scratch_bytes(M)));
    const int r = gemm_bf16(st, W_lm, V, H, X, M, EPI_HEAD, nullptr, 0, part, gemm_bf16_scratch_bytes(M) / sizeof(float),
                            cnt, tiles_for(M, V), nullptr, &p);
    if (r) return r == -4 ? EAGLE_ECUDA : EAGLE_EINVAL;
  } else {
    return EAGLE_EINVAL;
  }
  return head_merge(st, p) == 0 ? EAGLE_OK : EAGLE_ECUDA;
}

size_t eagle_op_attention_scratch_bytes(int R, int nq, int d) {
  if (R <= 0 || nq <= 0 || d <= 0) return 0;
  return al(attention_scratch_floats(R, nq, d) * sizeof(float));
}

int eagle_op_attention(int dtype, void* stream, const void* q, const void* kcache, const void* vcache, void* out, int R,
                       int nq, int nkv, int d, int cap, int rows_per_seq, const int32_t* row_seq,
                       const int32_t* row_slot, const int32_t* ctx_len, int mode, int tree_T, const uint64_t* mask,
                       int mask_words, float scale, int max_batch, void* scratch, size_t scratch_bytes) {
  if (!q || !kcache || !vcache || !out || !row_seq || !row_slot || !ctx_len || R <= 0 || nq <= 0 || nkv <= 0 ||
      d <= 0 || d > 128 || nq % nkv || rows_per_seq <= 0 || max_batch < 1 || (mode == 1 && (!mask || mask_words < 1)))
    return EAGLE_EINVAL;
  AttnArgs a{};
  a.q = q; a.kcache = kcache; a.vcache = vcache; a.out = out;
  a.R = R; a.nq = nq; a.nkv = nkv; a.d = d; a.cap = cap; a.rows_per_seq = rows_per_seq;
  a.row_seq = row_seq; a.row_slot = row_slot; a.ctx_len = ctx_len; a.mode = mode; a.tree_T = tree_T;
  a.mask = mask; a.mask_words = mask_words; a.scale = scale > 0.f ? scale : 1.f / sqrtf((float)d);
  if (scratch && scratch_bytes >= eagle_op_attention_scratch_bytes(R, nq, d)) {
    a.part_o = reinterpret_cast<float*>(scratch);
    a.part_floats = attention_scratch_floats(R, nq, d) / (d + 2) * d;
    a.part_ml = a.part_o + a.part_floats;
    a.max_splits = attention_max_splits(cap, max_batch);   // the engine's split policy for this cache
    a.kv_rows = (long long)max_batch * nkv * cap;
    a.max_batch = max_batch;
  } else if (dtype != EAGLE_DTYPE_F32) {
    return EAGLE_ECAPACITY;
  }
  const int r = attention(reinterpret_cast<cudaStream_t>(stream), dtype == EAGLE_DTYPE_F32 ? DT_F32 : DT_BF16, a);
  return r == 0 ? EAGLE_OK : (r == -1 ? EAGLE_EINVAL : EAGLE_ECUDA);
}

size_t eagle_op_tree_scratch_bytes(int B, int k, int depth, int m) {
  if (B < 1 || k < 1 || k > 16 || depth < 1 || depth > 8 || m < 1) return 0;
  const size_t NG = k + (size_t)(depth - 1) * k * k;
  const size_t T1 = m + 1;
  const size_t dmw = std::max<size_t>(1, ((depth - 1) * k + 63) / 64);
  size_t s = 0;
  s += al(B * NG * 4);                 // node_rank
  s += al((size_t)B * depth * k * 4);  // exp_node
  s += 7 * al((size_t)B * k * 4);      // drow_* (tok,pos,slot,seq,feat,plant) + head lse
  s += al((size_t)B * k * dmw * 8);    // dmask
  s += 3 * al(B * T1 * 4);             // tree_slot, tree_seq, margin
  s += al(B * T1 * k * 4);             // tree_kids
  s += 8 * al((size_t)B * 4);          // n_old, committed, on_track, cycle, acc_len, bonus, root_plant, spare
  s += 2 * al((size_t)B * k * k * 4);  // injected head rows of one depth (ids, values)
  return s;
}

int eagle_op_tree_build(void* stream, int B, int k, int depth, int m, const int32_t* cand_tok, const float* cand_logc,
                        const int32_t* child_tok, const float* child_logc, const int32_t* ctx_len,
                        const int32_t* root_tok, int32_t* node_tok, int32_t* node_parent, int32_t* node_depth,
                        float* node_logv, int32_t* tree_tok, int32_t* tree_pos, int32_t* tree_parent,
                        int32_t* tree_node, uint64_t* tree_mask, void* scratch, size_t scratch_bytes) {
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const size_t need = eagle_op_tree_scratch_bytes(B, k, depth, m);
  const int NG = k + (depth - 1) * k * k;
  if (!need || m > NG || !cand_tok || !cand_logc || !ctx_len || !root_tok || !node_tok || !node_parent ||
      !node_depth || !node_logv || !tree_tok || !tree_pos || !tree_parent || !tree_node || !tree_mask ||
      (depth > 1 && (!child_tok || !child_logc)))
    return EAGLE_EINVAL;
  if (!scratch || scratch_bytes < need) return EAGLE_ECAPACITY;
  const int T1 = m + 1;
  const int dmw = std::max(1, ((depth - 1) * k + 63) / 64);
  uint8_t* s = reinterpret_cast<uint8_t*>(scratch);
  auto take = [&](size_t bytes) { uint8_t* p = s; s += al(bytes); return p; };
  CycleDev c{};
  c.B = B; c.k = k; c.D = depth; c.m = m; c.T1 = T1; c.NG = NG; c.V = 0x7fffffff;
  c.dmask_words = dmw; c.tmask_words = (T1 + 63) / 64; c.fsrc_rows = 1 + (depth - 1) * k;
  c.ctx_len = const_cast<int*>(ctx_len);
  c.root_tok = const_cast<int*>(root_tok);
  c.kc = k;
  c.cand_tok = const_cast<int*>(cand_tok);
  c.cand_logc = const_cast<float*>(cand_logc);
  c.node_tok = node_tok; c.node_parent = node_parent; c.node_depth = node_depth; c.node_logv = node_logv;
  c.node_rank = (int*)take((size_t)B * NG * 4);
  c.exp_node = (int*)take((size_t)B * depth * k * 4);
  c.drow_tok = (int*)take((size_t)B * k * 4);
  c.drow_pos = (int*)take((size_t)B * k * 4);
  c.drow_slot = (int*)take((size_t)B * k * 4);
  c.drow_seq = (int*)take((size_t)B * k * 4);
  c.drow_feat = (int*)take((size_t)B * k * 4);
  c.drow_plant = (int*)take((size_t)B * k * 4);
  float* lse0 = (float*)take((size_t)B * k * 4);
  c.dmask = (uint64_t*)take((size_t)B * k * dmw * 8);
  c.tree_tok = tree_tok; c.tree_pos = tree_pos; c.tree_parent = tree_parent; c.tree_node = tree_node;
  c.tmask = tree_mask;
  c.tree_slot = (int*)take((size_t)B * T1 * 4);
  c.tree_seq = (int*)take((size_t)B * T1 * 4);
  c.margin = (float*)take((size_t)B * T1 * 4);
  c.tree_kids = (int*)take((size_t)B * T1 * k * 4);
  uint8_t* small = take(8 * al((size_t)B * 4)) ;
  c.n_old = (int*)small;
  c.committed = (int*)(small + al((size_t)B * 4));
  c.on_track = (int*)(small + 2 * al((size_t)B * 4));
  c.cycle = (uint32_t*)(small + 3 * al((size_t)B * 4));
  c.acc_len = (int*)(small + 4 * al((size_t)B * 4));
  c.bonus = (int*)(small + 5 * al((size_t)B * 4));
  c.root_plant = (int*)(small + 6 * al((size_t)B * 4));
  int* hid = (int*)take((size_t)B * k * k * 4);
  float* hval = (float*)take((size_t)B * k * k * 4);
  c.ref = nullptr;
  c.planted_p = 0.f;
  c.planted_conf = 0.5f;
  c.err = nullptr;
  if (cudaMemsetAsync(small, 0, 8 * al((size_t)B * 4), st) != cudaSuccess) return EAGLE_ECUDA;
  if (cudaMemsetAsync(lse0, 0, (size_t)B * k * 4, st) != cudaSuccess) return EAGLE_ECUDA;
  if (tree_start(st, c)) return EAGLE_ECUDA;
  for (int d = 1; d < depth; ++d) {
    if (tree_select(st, c, d)) return EAGLE_ECUDA;
    const size_t pitch = (size_t)(depth - 1) * k * k * 4;
    const size_t width = (size_t)k * k * 4;
    if (cudaMemcpy2DAsync(hid, width, child_tok + (size_t)(d - 1) * k * k, pitch, width, B, cudaMemcpyDeviceToDevice,
                          st) != cudaSuccess ||
        cudaMemcpy2DAsync(hval, width, child_logc + (size_t)(d - 1) * k * k, pitch, width, B,
                          cudaMemcpyDeviceToDevice, st) != cudaSuccess)
      return EAGLE_ECUDA;
    HeadOut h;
    h.top_id = hid; h.top_val = hval; h.lse = lse0; h.spec_logit = nullptr; h.K = k; h.S = 1;
    if (tree_add(st, c, d, h)) return EAGLE_ECUDA;
  }
  if (tree_finalize(st, c)) return EAGLE_ECUDA;
  return EAGLE_OK;
}

int eagle_op_compact(int dtype, void* stream, void* kcache, void* vcache, int layers, int B, int nkv, int cap, int d,
                     const int32_t* n_old, const int32_t* acc_len, const int32_t* acc_path, int Dmax) {
  if (!kcache || !vcache || !n_old || !acc_len || !acc_path || layers < 1 || B < 1 || nkv < 1 || d < 1 || Dmax < 1 ||
      Dmax > 8)
    return EAGLE_EINVAL;
  const int r = compact_kv(reinterpret_cast<cudaStream_t>(stream), dtype == EAGLE_DTYPE_F32 ? DT_F32 : DT_BF16, kcache,
                           vcache, layers, (size_t)B * nkv * cap * d, B, nkv, cap, d, n_old, acc_len, acc_path,
                           Dmax, KvPage{nullptr, 0, 0});
  return r == 0 ? EAGLE_OK : EAGLE_ECUDA;
}

}  // extern "C"
