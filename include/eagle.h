/*
 * eagle.h -- C ABI of the GB300 (sm_103a) EAGLE draft-and-verify cycle.
 *
 * One cycle, as the EAGLE pages define it:
 *   - feature-level drafting: the drafter embeds the one-step-advanced token,
 *     concatenates it with the target feature (EAGLE-1) or with g = FC([l; m; h]) of
 *     three target layers (EAGLE-3, its own output a replacing g on new draft
 *     positions), applies an FC and one decoder layer, and reuses the target's frozen
 *     embedding and LM head ("EAGLE: Feature-Level Drafting" lesson, sections "The big
 *     idea: draft at the feature level" and "Resolving the uncertainty by feeding back
 *     the token"; "EAGLE 三代" page, sections 2.3 and 4.3);
 *   - EAGLE-2 dynamic tree: path value = product of draft confidences, top-k
 *     expansion per depth, global top-m rerank, flattening with an ancestry mask
 *     ("EAGLE-2: Context-Aware Dynamic Draft Trees" page, sections "Path Value Ranks
 *     Prefixes", "Global Reranking", "The Mask Preserves Tree Semantics");
 *   - one tree-attention verify pass of the target over its KV cache;
 *   - lossless acceptance (greedy match, or rejection sampling along the tree) and
 *     compaction of the accepted path's KV entries (EAGLE lesson, "Speculative
 *     decoding in four moves"; EAGLE-2 page, table "Putting It Together", step 5).
 *
 * Conventions
 *   - Memory: weights, the workspace, inputs and outputs are caller-owned DEVICE
 *     memory. The library never allocates device memory; it carves everything it
 *     needs (KV caches, node tables, activations, scratch) out of the workspace.
 *     Host memory is used only for the context object and small host tables.
 *   - Streams: every call enqueues work on the context's stream and returns without
 *     waiting for the GPU (eagle_prefill reads its host length array; eagle_create
 *     and eagle_status_sync synchronise). Pass the stream as a cudaStream_t cast to
 *     void*. Graph replay (eagle_set_graph) needs a non-default stream.
 *   - Errors: every entry point returns an eagle_status. Host-detected problems are
 *     returned immediately with a message in eagle_last_error. Problems detected on
 *     the device (an out-of-range token or slot, a timed-out wait) are latched into a
 *     device status word and reported by eagle_status_sync. No kernel traps.
 *   - A context is not thread-safe.
 *
 * Weight layout (row-major, "out x in", storage type = dtype):
 *   embed [V][H], lm_head [V][H], final_norm [H]
 *   per layer: attn_norm [H], wqkv [(nq+2*nkv)*d][H] = [Wq; Wk; Wv],
 *              wo [H][nq*d], mlp_norm [H], wgu [2F][H] = [Wgate; Wup], wd [H][F]
 *   drafter kind 1: fc [H][2H] applied to [emb; f], then a layer shaped as above.
 *   drafter kind 3: fc [H][3H] applied to [l; m; h]; norm_g [H], norm_e [H];
 *              wqkv [(nq+2*nkv)*d][2H] applied to [RMSNorm(g); RMSNorm(emb)];
 *              wo, mlp_norm, wgu, wd as above (attn_norm unused).
 */
#ifndef EAGLE_H
#define EAGLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  EAGLE_OK = 0,
  EAGLE_EINVAL = -1,       /* bad argument or configuration */
  EAGLE_ECAPACITY = -2,    /* a length would exceed max_ctx / max_batch / the workspace */
  EAGLE_ECUDA = -3,        /* a CUDA runtime call or kernel launch failed */
  EAGLE_EDEVICE = -4,      /* a device-side check failed (bounds, capacity) */
  EAGLE_ETIMEOUT = -5,     /* a device-side wait exceeded its time limit */
  EAGLE_EUNSUPPORTED = -6  /* valid request this build does not implement */
} eagle_status;

enum { EAGLE_DTYPE_F32 = 0, EAGLE_DTYPE_BF16 = 1 };

typedef struct {
  int n_layers, hidden, n_heads, n_kv_heads, head_dim, ffn, vocab;
  float rope_theta, rms_eps;
  int dtype; /* EAGLE_DTYPE_F32 or EAGLE_DTYPE_BF16: storage and GEMM input type */
} eagle_model_cfg;

typedef struct {
  int kind;           /* 1 = EAGLE-1 feature drafter, 3 = EAGLE-3 fused drafter */
  int fuse_layers[3]; /* kind 3: 0-based target layers whose outputs are l, m, h */
} eagle_drafter_cfg;

typedef struct {
  int topk;           /* k: nodes expanded per depth and children per expanded node */
  int depth;          /* D: draft depths */
  int m;              /* nodes kept by the rerank (the verify pass scores m + 1 rows) */
  float temperature;  /* 0 = greedy, > 0 = speculative sampling at this temperature */
  uint64_t seed;      /* key of the counter-based (Philox4x32-10) draws */
  float planted_p;    /* planted-drafter probability per depth (0 = off) */
  float planted_conf; /* confidence given to a planted token */
} eagle_tree_cfg;

typedef struct {
  int max_batch;      /* sequences per context */
  int max_ctx;        /* KV entries per sequence (prompt + generated) */
  int kv_block;       /* 0 = contiguous target KV; 8..256 (a power of two) = paged target KV
                         in blocks of kv_block slots, assigned from a pool as sequences grow
                         (the drafter's one-layer cache stays contiguous) */
  int prefill_chunk;  /* prompt rows per prefill pass (0 = 512) */
} eagle_limits;

typedef struct {
  const void *attn_norm, *wqkv, *wo, *mlp_norm, *wgu, *wd;
} eagle_layer_weights;

typedef struct {
  const void *embed, *lm_head, *final_norm;
  const eagle_layer_weights* layers; /* host array of n_layers entries (copied) */
  const void *fc, *norm_g, *norm_e;  /* drafter input projections / EAGLE-3 norms */
  eagle_layer_weights draft;         /* the drafter's decoder layer */
} eagle_weights;

typedef struct eagle_ctx eagle_ctx;

/* Bytes of device workspace eagle_create needs for these configurations (0 on error). */
size_t eagle_workspace_bytes(const eagle_model_cfg* model, const eagle_drafter_cfg* drafter,
                             const eagle_tree_cfg* tree, const eagle_limits* limits);

/* Validate the configuration, carve `workspace` (ws_bytes >= eagle_workspace_bytes),
 * build the rotary tables (synchronous copy) and return a context in *out.
 * The weights must stay valid for the context's lifetime. */
int eagle_create(const eagle_model_cfg* model, const eagle_drafter_cfg* drafter, const eagle_tree_cfg* tree,
                 const eagle_weights* weights, const eagle_limits* limits, void* workspace, size_t ws_bytes,
                 void* stream, eagle_ctx** out);

/* Prefill `batch` prompts. d_tokens: device int32, prompts concatenated; h_lens: HOST
 * int32 [batch]. Runs the target over each prompt (causal), picks its first token
 * (greedy or sampled), runs the drafter over the prompt positions and prepares the
 * root's depth-1 candidates. d_ref (nullable): device int32 [batch][ref_len], the
 * target's own plain continuation of each prompt (its first entry being the prefill
 * token), which turns on planted-drafter mode (tree.planted_p). */
int eagle_prefill(eagle_ctx* ctx, int batch, const int32_t* d_tokens, const int32_t* h_lens,
                  const int32_t* d_ref, int ref_len);

/* Statistics of one cycle, written by the device into caller-owned device memory (8-byte
 * aligned) at the end of the cycle, stream-ordered like its outputs. The phases are the
 * cycle's steps ("EAGLE-2: Context-Aware Dynamic Draft Trees", table "Putting It Together",
 * steps 1-5): draft (the per-depth expansions and drafter passes), select (the global top-m
 * rerank, flattening and ancestry mask), verify (the target forward over the tree rows and
 * its LM-head epilogue), accept + compact (the acceptance walk and the KV compaction of the
 * accepted path), update (the drafter over the committed positions and the next root's
 * candidates). t_ns[0] is the device clock (%globaltimer, ns) once the work queued before
 * the cycle has finished; t_ns[i] (i = 1..5) once phase i's kernels have finished, so
 * t_ns[i] - t_ns[i - 1] is phase i's device time. */
typedef struct {
  int32_t batch;         /* sequences in the cycle (the prefilled batch) */
  int32_t active;        /* of them, those not finished before the cycle */
  int32_t accepted;      /* drafted tokens accepted, summed over the active sequences */
  int32_t committed;     /* tokens committed (accepted + bonus, cut at the limits), summed */
  int32_t max_accepted;  /* the longest accepted path */
  int32_t verify_rows;   /* tree rows verified per sequence (m + 1) */
  uint64_t t_ns[6];
} eagle_cycle_stats;

/* One draft-and-verify cycle for every sequence. d_out_tokens: device int32
 * [batch][depth + 1] receives the committed tokens (accepted path then the bonus
 * token); d_out_count: device int32 [batch] receives how many (L + 1); d_stats: device
 * eagle_cycle_stats (8-byte aligned). Any of them may be null; with d_stats the cycle
 * launches six one-thread clock kernels and one reduction more. Returns EAGLE_ECAPACITY,
 * before launching anything, when a sequence could outgrow max_ctx. The host-side enqueue
 * of each phase is an NVTX range ("eagle.cycle" around the call, "eagle.draft",
 * "eagle.select", "eagle.verify", "eagle.accept_compact", "eagle.update" inside; graph
 * replay enqueues nothing, so there only the outer range appears). */
int eagle_cycle(eagle_ctx* ctx, int32_t* d_out_tokens, int32_t* d_out_count, eagle_cycle_stats* d_stats);

/* Generation limits of the current batch: h_limits (HOST int32 [n], n = the prefilled
 * batch) gives each sequence's number of committed tokens, the prefill token included, at
 * which it is finished. A cycle that reaches a limit reports only the tokens up to it in
 * d_out_count (the surplus of its accepted path is dropped); a finished sequence is masked
 * out of every later cycle: d_out_count 0 and its state unchanged, while the others go on.
 * Its rows still pass through the cycle's fixed-shape launches. n = 0 removes the limits;
 * eagle_prefill removes them too. (The generation length is the pages' "new tokens" per
 * sequence; "EAGLE-2: Context-Aware Dynamic Draft Trees", table "Putting It Together".) */
int eagle_set_stop(eagle_ctx* ctx, int n, const int32_t* h_limits);

/* Draft budget between cycles: the next cycles expand `topk` nodes per depth (topk
 * children each) and keep m nodes, with 1 <= topk <= the created tree.topk and
 * 1 <= m <= min(the created tree.m, topk + (depth-1) topk^2). Takes effect at the next
 * eagle_cycle, in the middle of a generation: the root's candidates are always kept at the
 * created topk in rank order and the tree takes the first topk of them. The fixed k and m
 * of a tree stop fitting once the batch size changes what the GPU has to spare ("EAGLE-2:
 * Context-Aware Dynamic Draft Trees", table "Where It Breaks"); eagle_plan_budget
 * (eagle_ops.h) picks the pair this call applies. EAGLE_EINVAL while a static tree is set. */
int eagle_set_tree_budget(eagle_ctx* ctx, int topk, int m);

/* Plain (non-speculative) decoding of n_steps tokens per sequence from the current
 * state, one target pass per token: the lossless comparator and the speedup
 * baseline. d_out_tokens: device int32 [batch][n_steps]. d_out_margin (nullable):
 * device float [batch][n_steps], the top-2 logit margin of each greedy pick (NaN
 * when sampling), used to tell near-ties from real disagreements. */
int eagle_decode_plain(eagle_ctx* ctx, int n_steps, int32_t* d_out_tokens, float* d_out_margin);

/* Capture eagle_cycle into a CUDA graph on first use and replay it afterwards
 * (enable = 1), or launch kernels directly (enable = 0, the default). */
int eagle_set_graph(eagle_ctx* ctx, int enable);

/* Kernel launches one captured cycle replays (0 before the first captured cycle). */
int eagle_cycle_kernel_launches(const eagle_ctx* ctx);

/* Synchronise the context's stream and report latched device errors (clears them).
 * It also refreshes the host's bound on the sequences' KV lengths, which eagle_cycle
 * otherwise grows by depth + 1 per call to refuse cycles that could overflow. */
int eagle_status_sync(eagle_ctx* ctx);

/* Debug views: copy internal device state into the caller's device buffer `dst` of
 * `bytes` bytes (stream-ordered). Layouts (int32 unless noted, B = current batch):
 *   EAGLE_DUMP_STATE : ctx_len, root_tok, committed, on_track, cycle, acc_len, bonus  [7][B]
 *   EAGLE_DUMP_CAND  : cand_tok [B][k] int32, then cand_logc [B][k] float
 *   EAGLE_DUMP_NODES : tok, parent, depth [3][B][NG] int32, then logv [B][NG] float
 *                      (NG = k + (depth-1) k^2 nodes in generation order)
 *   EAGLE_DUMP_TREE  : tok, pos, parent, node [4][B][m+1] int32, then the ancestry
 *                      bitmask [B][m+1][ceil((m+1)/64)] uint64
 *   EAGLE_DUMP_ACCEPT: acc_len [B], bonus [B], acc_path [B][depth]
 *   EAGLE_DUMP_VERIFY_HEAD: top_id [B(m+1)][K] int32, top_val [B(m+1)][K] float,
 *                      lse [B(m+1)] float, child logits [B(m+1)][k] float
 *                      (K = 2 greedy, 1 sampling)
 *   EAGLE_DUMP_VERIFY_LOGITS: full verify logits [B(m+1)][V] float (only when
 *                      eagle_set_debug(ctx, EAGLE_DEBUG_LOGITS) was set before the cycle)
 *   EAGLE_DUMP_FEATURES: target features of the verify rows [B(m+1)][H] (storage type)
 *   EAGLE_DUMP_TTT   : after eagle_ttt_forward, its last step's R drafter outputs a
 *                      [R][H] (storage type), then each row's token cross-entropy [R]
 *                      float (R = the step's source rows; 0 bytes before any such call)
 * eagle_dump_bytes gives the size of each view. */
enum {
  EAGLE_DUMP_STATE = 0,
  EAGLE_DUMP_CAND = 1,
  EAGLE_DUMP_NODES = 2,
  EAGLE_DUMP_TREE = 3,
  EAGLE_DUMP_ACCEPT = 4,
  EAGLE_DUMP_VERIFY_HEAD = 5,
  EAGLE_DUMP_VERIFY_LOGITS = 6,
  EAGLE_DUMP_FEATURES = 7,
  EAGLE_DUMP_TTT = 8
};
size_t eagle_dump_bytes(const eagle_ctx* ctx, int what);
int eagle_debug_dump(eagle_ctx* ctx, int what, void* dst, size_t bytes);

enum { EAGLE_DEBUG_LOGITS = 1 };
int eagle_set_debug(eagle_ctx* ctx, int flags);

/* EAGLE-3 training-time-test forward (forward and loss only, no training), over one
 * sequence d_tokens (device int32 [n]): the target's causal pass gives every position's
 * drafter feature; drafter step 1 runs causally over sources t = 0..n-3 ([g_t; emb(x_{t+1})]
 * at position t); step s >= 2 feeds each source's previous output a back with x_{t+s}, at
 * position t+s-1, seeing the causal context up to t and its own earlier steps. d_loss
 * (device float [steps]) receives each step's mean cross-entropy of x_{t+s+1}. Requires
 * steps + 3 <= n <= prefill_chunk and n * steps within the drafter cache. It reuses sequence
 * 0's caches, so call eagle_prefill before the next eagle_cycle. */
int eagle_ttt_forward(eagle_ctx* ctx, const int32_t* d_tokens, int n, int steps, float* d_loss);

/* Static (EAGLE-1) tree policy: the same tree shape every cycle, fixed in advance, instead
 * of the EAGLE-2 dynamic tree. Host arrays of n = m nodes: parent[i] (-1 = a child of the
 * root, else an earlier node) and rank[i] in [0, k) (the drafter's rank[i]-th best child of
 * that parent). At most k nodes of one depth may have children; depth <= the draft depth.
 * The drafter still expands k rows per depth (the topology's nodes with children, then
 * others of that depth), and the verify pass scores exactly the topology. n = 0 restores
 * the dynamic tree. Synchronises the context's stream once (upload of two small tables). */
int eagle_set_static_tree(eagle_ctx* ctx, int n, const int32_t* parent, const int32_t* rank);

/* Device pointers of the target KV cache (storage type); for tests and tools. Contiguous
 * (kv_block = 0): layout [layer][batch][kv_head][slot][head_dim] with `cap` slots per sequence.
 * Paged: each layer is a pool [block][kv_head][slot in block][head_dim]; see eagle_kv_table. */
int eagle_kv_view(const eagle_ctx* ctx, void** k, void** v, int* cap);

/* Paged target KV: the device block table [batch][*tab_w] (int32, physical block of each
 * sequence's slots [j * kv_block, (j + 1) * kv_block), -1 = unassigned), the pool's blocks per
 * layer and the block size. EAGLE_EUNSUPPORTED for a contiguous cache. */
int eagle_kv_table(const eagle_ctx* ctx, const int32_t** table, int* tab_w, int* n_blocks, int* block);

/* Per-launch timing of the tensor-core GEMMs inside real cycles (graph replay off):
 * eagle_profile_begin arms CUDA events (host-created, no device allocation) around the
 * next max_launches GEMM launches (0: none, only the verify passes below are timed);
 * eagle_profile_end synchronises and returns the number of launches timed, their summed
 * device time (ms) and their algorithmic bytes (weight + activation input + output).
 * Events between launches stop the next kernel from starting before the previous one
 * ends, so time the verify pass in a window with max_launches = 0. */
int eagle_profile_begin(eagle_ctx* ctx, int max_launches);
int eagle_profile_end(eagle_ctx* ctx, int* launches, double* total_ms, double* total_bytes);

/* The verify passes (target forward over the tree rows + LM-head epilogue) of the cycles
 * run between eagle_profile_begin and eagle_profile_end (at most 64 are timed): how many
 * and their summed device time (CUDA events on the context's stream). */
int eagle_profile_verify(const eagle_ctx* ctx, int* passes, double* total_ms);

/* The same window's cycles phase by phase: how many cycles were timed and, in phase_ms[5],
 * each phase's summed device time (draft, select, verify, accept + compact, update; CUDA
 * events on the context's stream at the phase boundaries of eagle_cycle_stats). */
int eagle_profile_phases(const eagle_ctx* ctx, int* cycles, double* phase_ms);

const char* eagle_last_error(const eagle_ctx* ctx);
void eagle_destroy(eagle_ctx* ctx);

#ifdef __cplusplus
}
#endif
#endif /* EAGLE_H */
