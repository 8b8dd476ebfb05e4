// Host-side launchers of the cycle's CUDA kernels (internal to the library).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

struct HeadParams;

namespace eagle {

// Launch with programmatic stream serialization, so the kernel may begin launching while
// its predecessor finishes (each kernel calls griddepcontrol.wait before touching data).
// EAGLE_PDL=0 in the environment turns this off.
bool pdl_enabled();
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                     Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// EPI_GU: the [gate; up] projection in the paired tile layout of EPI_SWIGLU (64 gate + the
// matching 64 up features per tile), storing fp32 gate and up values to out [M][2N] (gate
// at f, up at N + f); a separate SwiGLU pass over them then gives the fused epilogue's bits.
enum { EPI_F32 = 0, EPI_BF16 = 1, EPI_ADD_F32 = 2, EPI_HEAD = 3, EPI_SWIGLU = 4, EPI_QKV = 5, EPI_GU = 6 };

// EPI_QKV: the fused [q | k | v] projection's epilogue applies rotate-half RoPE to the q and
// k heads (pairs inside one 128-row tile: head_dim divides 128), writes q to its buffer
// [R][nq][d] and k, v into the cache at each row's slot (storage bf16).
struct QkvEpi {
  const int* pos;
  const int* slot;
  const int* seq;
  const float* cos;       // [positions][d / 2]
  const float* sin;
  void* q;
  void* kc;               // [(seq * nkv + h) * cap + slot][d]
  void* vc;
  int nq, nkv, d, cap;
};
enum { DT_F32 = 0, DT_BF16 = 1 };

inline int num_sms_cap() { return 192; }
// SM count of the current device (cached per device).
int device_sm_count();
// Raise a kernel's dynamic shared-memory limit on the current device to at least `bytes`
// (the limit is only ever raised, so launches of any smaller size stay valid).
cudaError_t raise_smem_limit(const void* func, int bytes);

// ---- GEMMs -------------------------------------------------------------------------------
int gemm_bn_for(int M);
// partial-sum scratch of GEMMs of up to max_rows rows
size_t gemm_bf16_scratch_bytes(int max_rows);
// bf16 tcgen05 GEMM, Y[M][N] = X[M][K] W[N][K]^T. Returns 0 or a negative code (-2: the
// counters or the partial-sum scratch are too small for this shape).
int gemm_bf16(cudaStream_t st, const void* W, int N, int K, const void* X, int M, int epi, void* out,
              int ldo, float* partials, size_t partial_floats, int* counters, int counters_len, int* err,
              const HeadParams* head, bool cache_maps = true, const QkvEpi* qkv = nullptr);
// EPI_SWIGLU: W is [2N][K] ([gate; up]), out bf16 [M][ldo] = silu(X Wg^T) * (X Wu^T); N % 64 == 0.
// Tensor map of a bf16 row-major [rows][K] matrix (row stride ld elements, 0 = K): boxes of
// 64 (K) x box_rows, 128-byte swizzle. Cached by (ptr, rows, K, box_rows, ld).
bool make_tmap_bf16(CUtensorMap* m, const void* ptr, long long rows, long long K, int box_rows, long long ld = 0);
// fp32 SIMT GEMM with the same contract (EPI_F32 / EPI_ADD_F32).
int gemm_f32(cudaStream_t st, const float* W, int N, int K, const float* X, int M, int epi, float* out,
             int ldo);

// ---- LM head reductions ------------------------------------------------------------------
// Partial records from materialised logits [n_rows][ld] (fp32 path).
int head_partials_from_logits(cudaStream_t st, const float* logits, int ld, const HeadParams& p);
int head_merge(cudaStream_t st, const HeadParams& p);
size_t head_part_bytes(int vocab, int rows, int K);

// ---- KV-cache addressing ----------------------------------------------------------------------
// Contiguous cache (table == nullptr): one layer is [seq][nkv][cap][d]. Paged cache: one layer
// is a pool of blocks of 2^bs_log2 token slots, [block][nkv][slot in block][d], and
// table[seq * tab_w + j] is the physical block that holds the sequence's slots
// [j << bs_log2, (j + 1) << bs_log2) (-1 = not assigned yet).
struct KvPage {
  const int* table;
  int tab_w;
  int bs_log2;
};
// Row (in units of d elements) of key/value head h of sequence seq at slot.
__host__ __device__ inline size_t kv_row(const KvPage& p, int seq, int nkv, int h, int cap, int slot) {
  if (!p.table) return ((size_t)seq * nkv + h) * (size_t)cap + (size_t)slot;
  int blk = p.table[(size_t)seq * p.tab_w + (slot >> p.bs_log2)];
  if (blk < 0) blk = 0;   // unassigned: writers check first; a read stays inside the pool
  return (((size_t)blk * nkv + h) << p.bs_log2) + (size_t)(slot & ((1 << p.bs_log2) - 1));
}

// ---- element-wise / row ops (dtype = DT_F32 or DT_BF16 storage) --------------------------
int embed_rows(cudaStream_t st, int dtype, const void* E, int V, int H, const int* tok, int R, float* x,
               int* err);
// EAGLE-3 drafter input (bf16): gather of the feature rows, fp32 residual, [RMSNorm(g) * norm_g;
// RMSNorm(emb) * norm_e] in one pass per row.
int eagle3_input_rows(cudaStream_t st, const void* feat, const int* feat_row, const void* E, int V, const int* tok,
                      int H, const void* norm_g, const void* norm_e, float eps, void* gbuf, float* x, void* ebuf,
                      void* ain, int R, int* err);
int rmsnorm_rows(cudaStream_t st, int dtype_in, const void* x, int ldx, const void* g, int H, float eps,
                 int R, int dtype_out, void* out, int ldo);
int rope_store(cudaStream_t st, int dtype, const float* qkv, int R, int nq, int nkv, int d,
               const int* row_pos, const int* row_slot, const int* row_seq, const float* rope_cos,
               const float* rope_sin, void* q_out, void* kcache, void* vcache, int cap, int* err, int slot_limit,
               const KvPage& page = KvPage{nullptr, 0, 0});
int swiglu_rows(cudaStream_t st, int dtype, const float* gu, int F, int R, void* out);
int concat_emb_feat(cudaStream_t st, int dtype, const void* E, int V, int H, const int* tok,
                    const void* feat, const int* feat_row, int R, void* out, int* err);
int convert_rows(cudaStream_t st, int dtype, const float* x, int H, int R, void* out, int ldo);
// dst row (dst_idx ? dst_idx[r] : r) <- src row (idx ? idx[r] : r). With src_rows > 0 a source
// index outside [0, src_rows) is latched into *err (DEVERR_BOUNDS) and its row skipped.
int gather_rows(cudaStream_t st, size_t row_bytes, const void* src, size_t src_ld, const int* idx, int R,
                void* dst, size_t dst_ld, const int* dst_idx = nullptr, int src_rows = 0, int* err = nullptr);
int widen_rows(cudaStream_t st, int dtype, const void* x, int ldx, int H, int R, float* out);

// ---- attention -----------------------------------------------------------------------------
struct AttnArgs {
  const void* q;        // [R][nq][d]
  const void* kcache;   // this layer: row kv_row(page, seq, nkv, h, cap, slot) of d elements
  const void* vcache;
  KvPage page;          // table == nullptr: contiguous [(seq * nkv + h) * cap + slot][d]
  void* out;            // [R][nq][d]
  int R, nq, nkv, d, cap;
  int rows_per_seq;     // rows of one sequence are contiguous; a row block never straddles two
  const int* row_seq;   // [R]
  const int* row_slot;  // [R]  slot of the row's own key
  const int* ctx_len;   // [B] slots [0, ctx_len) are visible to every row of the sequence
  int mode;             // 0 = causal (slot <= row_slot), 1 = tree (ctx + mask bits over slots ctx..ctx+T),
                        // 2 = training-time test (n = ctx_len; see attention.cu)
  int tree_T;
  const uint64_t* mask; // [R][mask_words]
  int mask_words;
  float scale;
  // scratch of the tensor-core path (bf16, required): each key split's partial outputs and
  // (max, sum) pairs, merged with the row's tail in a fixed order
  float* part_o;        // [splits][R][nq][d]
  float* part_ml;       // [splits][R][nq][2]
  size_t part_floats;   // capacity of part_o in floats (the number of key splits is capped to fit)
  int* err;             // device status word for bounds checks (nullable)
  int max_splits;       // key splits of the bf16 path (1..32): a constant of the caller, so that
                        // every launch over one cache sums a row's keys in the same splits
  long long kv_rows;    // rows of d elements in the cache buffers (their TMA extent; 0: unknown,
                        // the bf16 path then stays on mma.sync)
  int max_batch;        // sequences the caller's engine serves (a constant of the engine)
};
int attention(cudaStream_t st, int dtype, const AttnArgs& a);
size_t attention_scratch_floats(int rows, int nq, int d);
// the key splits to use for a cache of `cap` slots (one 64-key tile per split, up to 31);
// the partial buffer needs one more slot per row for the tail
int attention_max_splits(int cap, int batch);

// ---- tree policy, acceptance, compaction ---------------------------------------------------
struct TreeState;   // defined in tree.cu / engine
}  // namespace eagle
