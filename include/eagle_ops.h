/*
 * eagle_ops.h -- kernel-level entry points of the EAGLE cycle library.
 *
 * Each call runs one of the cycle's kernels on caller-provided device buffers, so it
 * can be checked on its own against the CPU oracle with injected inputs. All pointers
 * are DEVICE pointers unless stated; `stream` is a cudaStream_t cast to void*; calls
 * are stream-ordered and return an eagle_status (see eagle.h) without waiting.
 * `scratch` is caller-owned device memory of at least the size the matching
 * *_scratch_bytes function returns; the library never allocates device memory.
 */
#ifndef EAGLE_OPS_H
#define EAGLE_OPS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Projection GEMM Y[M][N] = X[M][K] * W[N][K]^T (the nn.Linear layout used for every
 * target and drafter projection and the LM head). dtype EAGLE_DTYPE_BF16: tcgen05
 * tensor-core kernel, X and W bf16 row-major with K a multiple of 8 and 16-byte
 * aligned bases; dtype EAGLE_DTYPE_F32: fp32 FFMA kernel. epi: 0 = store fp32 Y,
 * 1 = store bf16 Y (bf16 only), 2 = Y += result (fp32 residual update), 4 = SwiGLU
 * (bf16 only, N % 64 == 0): W holds 2N rows [Wgate; Wup] and out (bf16, [M][N]) receives
 * silu(X Wgate^T) * (X Wup^T); size its scratch with eagle_op_gemm_scratch_bytes(M, 2N).
 * out has row stride ldo elements. Scratch holds split-tile partial sums and per-tile
 * counters; it must be zero-filled before the first call and is left zeroed by every call.
 * The kernel's CTAs hand partial sums to one another, so no other work may hold SMs for
 * the whole of a call (kernels on other streams that finish on their own are fine). */
size_t eagle_op_gemm_scratch_bytes(int M, int N);
int eagle_op_gemm(int dtype, void* stream, const void* W, int N, int K, const void* X, int M, int epi,
                  void* out, int ldo, void* scratch, size_t scratch_bytes);

/* Allocation-free variant of eagle_op_gemm (bf16 only) for callers that cannot
 * allocate device memory where they run a projection, e.g. plugins of a host framework
 * that hands them only input and output buffers, or runtimes that pool all device
 * memory in advance. The paper has no counterpart: this is a deployment convenience.
 * Its split-tile scratch lives in file-scope device arrays of the library (about 6 MiB
 * on every GPU that loads it, held until the process exits), so the call allocates
 * nothing (no cudaMalloc/cudaFree, no allocating library routine).
 * Limits: M <= 32 rows and at most 8192 output tiles (ceil(N/128) tiles for M <= 32);
 * larger requests return EAGLE_ECAPACITY. epi as eagle_op_gemm (0, 1 or 2).
 * The first call on a device looks up the arrays' device addresses (cudaGetSymbolAddress)
 * with that device current; make that first call before any stream capture. All calls
 * share the one scratch area and the last call's contents remain in it: calls that may
 * overlap on the GPU (different streams without ordering) race and must not be issued;
 * graph replays that contain this call must be serialised the same way.
 * A bounded device wait that gives up leaves `out` incomplete and records a timeout in a
 * status word that is also a file-scope device array; read it with
 * eagle_op_gemm_noalloc_status. */
int eagle_op_gemm_noalloc(void* stream, const void* W, int N, int K, const void* X, int M, int epi, void* out,
                          int ldo);

/* Status of the allocation-free GEMM on the current device: waits for `stream`, reads
 * the status word that its calls share and clears it. EAGLE_OK when no call since the
 * last read gave up, EAGLE_ETIMEOUT when one did (its output is incomplete). */
int eagle_op_gemm_noalloc_status(void* stream);

/* Fused LM head: logits = X[M][H] * W_lm[V][H]^T reduced per row without writing the
 * logits (bf16), or through an fp32 logits buffer inside the scratch (f32). Per row it
 * returns the K best entries by ranking value (value desc, token id asc) and the
 * log-sum-exp of logit * inv_t. Ranking value = logit * inv_t, plus Gumbel(0,1) noise
 * when gumbel != 0, drawn from Philox4x32-10 keyed by (seed; counter = (id >> 2,
 * row_key[row], cycle, row_seq[row] << 8 | stream_id)), word id & 3. specials
 * [M][S] (nullable, -1 = unused): ids left out of the ranking (and out of the
 * log-sum-exp when lse_excl != 0) whose raw logits go to spec_logit [M][S].
 * Outputs: top_id [M][K] int32, top_val [M][K] float, lse [M] float. K in 1..16. */
size_t eagle_op_lm_head_scratch_bytes(int dtype, int V, int M, int K);
int eagle_op_lm_head(int dtype, void* stream, const void* W_lm, int V, int H, const void* X, int M, int K,
                     float inv_t, int gumbel, int lse_excl, const int32_t* specials, int S, float* spec_logit,
                     const int32_t* row_seq, const int32_t* row_key, uint32_t cycle, uint64_t seed,
                     int stream_id, int32_t* top_id, float* top_val, float* lse, void* scratch,
                     size_t scratch_bytes);

/* Tree-masked attention of R query rows over a KV cache laid out
 * [seq][kv_head][slot][d] with `cap` slots and max_batch sequences (storage type dtype;
 * row_seq < max_batch). q, out: [R][nq][d].
 * Rows of one sequence are contiguous, rows_per_seq each; row r belongs to sequence
 * row_seq[r] and its own key sits at slot row_slot[r]. mode 0 (causal): row r sees
 * slots <= row_slot[r]. mode 1 (tree): row r sees slots < ctx_len[seq] and slot
 * ctx_len[seq] + t for t < tree_T where bit t of mask[r][t / 64] is set.
 * Scale = 1/sqrt(d) when scale <= 0. fp32: d <= 128, scratch unused (nullable); bf16
 * (tensor cores): d in {32, 64, 128}, 64 divisible by nq/nkv, tree_T <= 256, scratch of
 * eagle_op_attention_scratch_bytes required (EAGLE_ECAPACITY without it). The bf16 path
 * gives each row a result that does not depend on the other rows of the call: a row at
 * logical position P (its own slot in causal mode, ctx_len + its mask's popcount - 1 in
 * tree mode, whose ancestors must have increasing slots by depth) has its keys up to
 * position P - 16 summed in fixed key splits on the tensor cores, its last 16 positions in
 * position order on the FMA units, and the two merged in a fixed order; so a tree row and
 * a causal row at the same position over the same keys give bit-identical outputs. The
 * split length is that of an engine serving up to max_batch sequences (>= 1): three
 * 64-key tiles below eight sequences, eight from eight on; calls with the same cap and
 * max_batch share it. With d = 128 and EAGLE_ATTN_TC=1 in the environment the splits run on
 * tcgen05 (TMA tiles of the cache, S and O in TMEM; a different summation order, fixed for the
 * process). */
size_t eagle_op_attention_scratch_bytes(int R, int nq, int d);
int eagle_op_attention(int dtype, void* stream, const void* q, const void* kcache, const void* vcache,
                       void* out, int R, int nq, int nkv, int d, int cap, int rows_per_seq,
                       const int32_t* row_seq, const int32_t* row_slot, const int32_t* ctx_len, int mode,
                       int tree_T, const uint64_t* mask, int mask_words, float scale, int max_batch,
                       void* scratch, size_t scratch_bytes);

/* EAGLE-2 tree growth and rerank with injected draft confidences, for B sequences:
 * cand_tok/cand_logc [B][k]: the root's children (token, log confidence) in rank order;
 * child_tok/child_logc [B][depth-1][k][k]: children of the r-th node selected at depth
 * d (entry [b][d-1][r][i], rank order). ctx_len [B], root_tok [B].
 * Outputs: node tables [B][NG] (tok, parent, depth int32; logv float), flattened tree
 * [B][m+1] (tok, pos, parent, node int32) and ancestry bitmask [B][m+1][W] uint64 with
 * W = ceil((m+1)/64). */
size_t eagle_op_tree_scratch_bytes(int B, int k, int depth, int m);
int eagle_op_tree_build(void* stream, int B, int k, int depth, int m, const int32_t* cand_tok,
                        const float* cand_logc, const int32_t* child_tok, const float* child_logc,
                        const int32_t* ctx_len, const int32_t* root_tok, int32_t* node_tok, int32_t* node_parent,
                        int32_t* node_depth, float* node_logv, int32_t* tree_tok, int32_t* tree_pos,
                        int32_t* tree_parent, int32_t* tree_node, uint64_t* tree_mask, void* scratch,
                        size_t scratch_bytes);

/* KV compaction: in every layer, slot n_old[b] + j <- slot n_old[b] + acc_path[b][j-1]
 * for j = 1..acc_len[b] (acc_path rows are flattened-tree rows, Dmax per sequence,
 * Dmax <= 8). Cache layout [layer][seq][kv_head][slot][d], cap slots per sequence. */
int eagle_op_compact(int dtype, void* stream, void* kcache, void* vcache, int layers, int B, int nkv, int cap,
                     int d, const int32_t* n_old, const int32_t* acc_len, const int32_t* acc_path, int Dmax);

/* Batch-aware draft budget (host arithmetic only, no device work). For each candidate k
 * (k_values[j], n_k of them) the caller supplies draft_us[j], the measured drafter cost of a
 * cycle, and exp_tokens[off_j + m - 1] for m = 1..m_max[j] (off_j = sum of the earlier
 * m_max), the expected committed tokens per sequence of a tree of m nodes: 1 + the sum of
 * the m largest path values, averaged over real cycles (a node's path value estimates its
 * acceptance: "EAGLE-2: Context-Aware Dynamic Draft Trees", "Path Value Ranks Prefixes").
 * rows_pts / verify_us (n_points, rows strictly increasing) are measured verify-pass times
 * against verify rows; between points the time is interpolated linearly, beyond the last
 * it grows with the last slope (flat before the first; a single point is flat up to it and
 * proportional past it). Returns in best_k / best_m the choice maximising
 * batch * exp_tokens / (draft_us + verify(batch * (m + 1))) and that rate (tokens per
 * microsecond, nullable). Ties keep the earlier k and the smaller m. EAGLE_EINVAL on bad
 * arguments. */
int eagle_plan_budget(int n_k, const int32_t* k_values, const float* draft_us, const int32_t* m_max,
                      const float* exp_tokens, int n_points, const int32_t* rows_pts, const float* verify_us,
                      int batch, int32_t* best_k, int32_t* best_m, float* tokens_per_us);

/* Failure-detection probe. Runs one of the library's bounded device waits on a condition
 * that nothing satisfies and returns once it gives up: kind 0 waits on a shared-memory
 * mbarrier phase that nobody completes (the wait of the TMA / tensor-core pipelines),
 * kind 1 waits until the device word *d_counter (caller-owned, zero, nullable for kind 0)
 * reaches 1 (the wait of the split-tile owner). Each wait stops after
 * the library's limit of 2 s of %globaltimer and atomically latches 1 (timeout) into *d_err
 * if it is still 0; *d_result receives 1 if the wait was satisfied, 0 if it gave up. Launches
 * one CTA on `stream` and returns without synchronising; EAGLE_EINVAL on a bad kind or a
 * null pointer. */
int eagle_op_wait_probe(void* stream, int kind, const unsigned* d_counter, int* d_err, int* d_result);

#ifdef __cplusplus
}
#endif
#endif /* EAGLE_OPS_H */
