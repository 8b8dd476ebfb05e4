// Cycle orchestrator and C ABI (eagle.h).
//
// The engine owns no device memory: it carves the caller's workspace into KV caches,
// node tables, activations and scratch, and enqueues the kernels of prefill, the
// draft-and-verify cycle and plain decoding on one stream. The cycle has a fixed launch
// sequence (D - 1 drafter expansions, one verify pass over m + 1 rows per sequence, an
// update pass padded to D + 1 rows), with every data-dependent quantity (accepted
// length, positions, slots) read from device memory, so it can be captured once in a
// CUDA graph and replayed.
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <algorithm>
#include <climits>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "../../include/eagle.h"
#include "common.cuh"
#include "cycle.h"
#include "kernels.h"
#include "lmhead.cuh"

using namespace eagle;

namespace eagle {
int root_candidates_seq(cudaStream_t st, const CycleDev& c, const HeadOut& h, int seq);
}

namespace {

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Carver {
  uint8_t* base = nullptr;
  size_t off = 0;
  template <typename T>
  T* take(size_t count) {
    off = align_up(off, 256);
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += count * sizeof(T) + 16;
    return p;
  }
};

struct Dims {
  int L, H, F, V, nq, nkv, d, QKV, A, B, k, D, m, T1, NG, cap, dcap, P, Rt, Rd, R, Rh, KIN, fsrc_rows, dmw, tmw,
      rope_pos, kind, esz, dt, max_ctx, n_tiles, Kh;
  // target KV cache: kvb_log2 = 0 contiguous, else blocks of 2^kvb_log2 slots, tab_w blocks
  // per sequence in the block table, nblk blocks in the pool; kv_layer_elems per layer
  int kvb_log2, tab_w, nblk;
  size_t kv_layer_elems;
};

bool derive(const eagle_model_cfg* mc, const eagle_drafter_cfg* dc, const eagle_tree_cfg* tc,
            const eagle_limits* lim, Dims& z, std::string& why) {
  if (!mc || !dc || !tc || !lim) { why = "null configuration"; return false; }
  z.L = mc->n_layers; z.H = mc->hidden; z.F = mc->ffn; z.V = mc->vocab;
  z.nq = mc->n_heads; z.nkv = mc->n_kv_heads; z.d = mc->head_dim;
  if (z.L <= 0 || z.H <= 0 || z.F <= 0 || z.V <= 0 || z.nq <= 0 || z.nkv <= 0 || z.d <= 0) { why = "model sizes must be positive"; return false; }
  if (z.nq % z.nkv) { why = "n_heads must be a multiple of n_kv_heads"; return false; }
  if (z.d > 128 || (z.d % 2)) { why = "head_dim must be even and <= 128"; return false; }
  if (mc->dtype != EAGLE_DTYPE_F32 && mc->dtype != EAGLE_DTYPE_BF16) { why = "dtype must be f32 or bf16"; return false; }
  z.dt = mc->dtype == EAGLE_DTYPE_F32 ? DT_F32 : DT_BF16;
  z.esz = z.dt == DT_F32 ? 4 : 2;
  z.QKV = (z.nq + 2 * z.nkv) * z.d;
  z.A = z.nq * z.d;
  if (z.dt == DT_BF16 && ((z.H % 8) || (z.F % 8) || (z.A % 8))) { why = "bf16 GEMM sizes must be multiples of 8"; return false; }
  z.kind = dc->kind;
  if (z.kind != 1 && z.kind != 3) { why = "drafter kind must be 1 or 3"; return false; }
  if (z.kind == 3)
    for (int i = 0; i < 3; ++i)
      if (dc->fuse_layers[i] < 0 || dc->fuse_layers[i] >= z.L) { why = "fuse_layers out of range"; return false; }
  z.k = tc->topk; z.D = tc->depth; z.m = tc->m;
  if (z.k < 1 || z.k > 16) { why = "topk must be in 1..16"; return false; }
  if (z.D < 1 || z.D > 8) { why = "depth must be in 1..8"; return false; }
  z.NG = z.k + (z.D - 1) * z.k * z.k;
  if (z.m < 1 || z.m > z.NG || z.m + 1 > 256) { why = "m must be in 1..min(N_gen, 255)"; return false; }
  if (tc->temperature < 0.f) { why = "temperature must be >= 0"; return false; }
  if (tc->planted_p < 0.f || tc->planted_p > 1.f || tc->planted_conf <= 0.f || tc->planted_conf >= 1.f) {
    why = "planted_p must be in [0,1] and planted_conf in (0,1)"; return false; }
  if (lim->max_batch < 1 || lim->max_ctx < 2) { why = "max_batch >= 1 and max_ctx >= 2 required"; return false; }
  if (lim->kv_block < 0 || (lim->kv_block != 0 && (lim->kv_block < 8 || lim->kv_block > 256 ||
                                                    (lim->kv_block & (lim->kv_block - 1))))) {
    why = "kv_block must be 0 (contiguous KV) or a power of two in 8..256"; return false; }
  z.B = lim->max_batch;
  z.max_ctx = lim->max_ctx;
  z.T1 = z.m + 1;
  z.cap = z.max_ctx + z.T1 + 8;
  z.dcap = z.max_ctx + std::max((z.D - 1) * z.k, z.D + 1) + 8;
  z.P = lim->prefill_chunk > 0 ? lim->prefill_chunk : 512;
  if (z.P > z.max_ctx) z.P = z.max_ctx;
  z.Rt = std::max(std::max(z.B * z.T1, z.P), z.B);
  z.Rd = std::max(std::max(z.B * z.k, z.B * (z.D + 1)), z.P);
  z.R = std::max(z.Rt, z.Rd);
  z.Rh = std::max(std::max(z.B * z.T1, z.B * z.k), z.B);
  z.KIN = std::max(std::max(3 * z.H, z.A), z.F);
  z.fsrc_rows = 1 + (z.D - 1) * z.k;
  z.dmw = std::max(1, ((z.D - 1) * z.k + 63) / 64);
  z.tmw = (z.T1 + 63) / 64;
  z.rope_pos = std::max(z.cap, z.dcap) + 8;
  z.n_tiles = (z.V + 127) / 128;
  z.Kh = std::max(z.k, 2);
  z.kvb_log2 = 0;
  while (lim->kv_block > 0 && (1 << z.kvb_log2) < lim->kv_block) ++z.kvb_log2;
  if (z.kvb_log2 > 0) {
    z.tab_w = (z.cap + lim->kv_block - 1) >> z.kvb_log2;
    z.nblk = z.B * z.tab_w;
    z.kv_layer_elems = (size_t)z.nblk * z.nkv * ((size_t)1 << z.kvb_log2) * z.d;
  } else {
    z.tab_w = 0;
    z.nblk = 0;
    z.kv_layer_elems = (size_t)z.B * z.nkv * z.cap * z.d;
  }
  return true;
}

constexpr int PHASES = 5;   // draft, select, verify, accept + compact, drafter update

}  // namespace

struct eagle_ctx {
  Dims z;             // current dimensions (k and m may be lowered between cycles)
  Dims zc;            // dimensions at creation: the workspace is carved for these
  eagle_model_cfg mc;
  eagle_drafter_cfg dc;
  eagle_tree_cfg tc;
  eagle_limits lim;
  eagle_weights w;
  std::vector<eagle_layer_weights> layers;
  cudaStream_t st = nullptr;
  std::string err;
  int batch = 0;
  long long host_ctx_bound = 0;   // upper bound of every sequence's KV length
  int ref_len = 0;
  int graph_enabled = 0;
  cudaGraphExec_t graph = nullptr;
  const int32_t* graph_out = nullptr;   // output pointers baked into the captured graph
  const int32_t* graph_cnt = nullptr;
  const int32_t* graph_ref = nullptr;
  int graph_batch = 0;
  int graph_kernels = 0;                // kernel nodes of the captured cycle
  int debug = 0;
  // per-launch GEMM profiling (events around every tensor-core GEMM launch)
  std::vector<cudaEvent_t> prof_ev;
  std::vector<double> prof_bytes;
  int prof_on = 0, prof_n = 0;
  // profiled cycles: events at the cycle's start and at the end of each of its five phases
  std::vector<cudaEvent_t> ph_ev;       // [64][PHASES + 1]
  int ph_n = 0, ph_done = 0;            // cycles recorded / timed by eagle_profile_end
  double ph_ms[PHASES] = {0, 0, 0, 0, 0};
  // cycle statistics: the caller's struct baked into the captured graph
  eagle_cycle_stats* graph_stats = nullptr;
  eagle_cycle_stats* stats = nullptr;   // of the cycle being enqueued (null: none)
  // buffers
  int* dev_err;
  int *ctx_len, *n_old, *root_tok, *committed, *on_track, *root_plant, *acc_len, *bonus, *acc_path, *root_row, *iota;
  int* emitted;       // [B] tokens the last cycle committed for each sequence (0: finished)
  int* stop_at;       // [B] committed-token limit of each sequence (INT32_MAX: none)
  uint32_t *cycle, *plain_step;
  int *cand_tok; float* cand_logc;
  int *node_tok, *node_parent, *node_depth, *node_rank, *exp_node; float* node_logv;
  int *drow_tok, *drow_pos, *drow_slot, *drow_seq, *drow_feat, *drow_plant, *drow_out; uint64_t* dmask;
  int *tree_tok, *tree_pos, *tree_slot, *tree_seq, *tree_parent, *tree_node, *tree_kids; uint64_t* tmask; float* margin;
  int *row_tok, *row_pos, *row_slot, *row_seq, *row_feat;
  float *x, *qkv, *gu;
  void *ain, *qb, *att, *hb, *feat_t, *caps, *dout, *fsrc, *gbuf, *ebuf, *pre_feat;
  float* logits;
  float *h_part, *h_val, *h_lse, *h_spec; int* h_id;        // drafter / root / plain heads
  float *v_val, *v_lse, *v_spec, *v_logits; int* v_id;       // verify head (kept for the cycle's dump)
  float* gemm_part; size_t gemm_part_floats; int* gemm_cnt; int gemm_cnt_len;
  float *attn_po, *attn_pml; size_t attn_pfloats;
  // bf16 fused epilogues, the bits of EAGLE_FUSE_EPI: 1 = SwiGLU in the gate/up epilogue
  // (the default: measured faster at every batch, 8B batch-1 verify 4.61 -> 4.57 ms),
  // 2 = RoPE/KV write in the QKV epilogue (slower at 61 rows: 4.96 ms), at every row count
  // (0: none, 3: both; -1: SwiGLU from 128 rows on). Both epilogues agree bit for bit with
  // the row kernels they replace.
  int fuse_epi = 1;
  float *rope_cos, *rope_sin;
  void *kc, *vc, *dkc, *dvc;
  int *static_exp, *static_keep;        // static tree: [D-1][k] expansion rows, [NG] kept flags
  int static_on = 0;
  std::vector<int> h_static_exp, h_static_keep;
  int* ttt_tgt;       // training-time test: the target token of each row
  float* ttt_acc;     // training-time test: running loss sum
  float* ttt_ce;      // training-time test: the last step's per-row cross-entropy
  int ttt_rows = 0;   // rows of the last training-time-test step (0: none run yet)
  int* kv_table;      // paged target KV: [B][tab_w] physical block per logical block, -1 = none
  int* kv_next;       // next free block of the pool (one device counter)
  KvPage page;        // the target cache's addressing (table == nullptr: contiguous)
  int* prompt_copy;   // unused placeholder
  CycleDev cd;
};

namespace {

void carve(Carver& c, eagle_ctx* x, const Dims& z) {
  const int B = z.B;
  x->dev_err = c.take<int>(4);
  x->ctx_len = c.take<int>(B); x->n_old = c.take<int>(B); x->root_tok = c.take<int>(B);
  x->committed = c.take<int>(B); x->on_track = c.take<int>(B); x->root_plant = c.take<int>(B);
  x->acc_len = c.take<int>(B); x->emitted = c.take<int>(B); x->bonus = c.take<int>(B); x->acc_path = c.take<int>((size_t)B * z.D);
  x->root_row = c.take<int>(B); x->iota = c.take<int>(std::max(B, z.R));
  x->stop_at = c.take<int>(B);
  x->cycle = c.take<uint32_t>(B); x->plain_step = c.take<uint32_t>(4);
  x->cand_tok = c.take<int>((size_t)B * z.k); x->cand_logc = c.take<float>((size_t)B * z.k);
  x->node_tok = c.take<int>((size_t)B * z.NG); x->node_parent = c.take<int>((size_t)B * z.NG);
  x->node_depth = c.take<int>((size_t)B * z.NG); x->node_rank = c.take<int>((size_t)B * z.NG);
  x->node_logv = c.take<float>((size_t)B * z.NG); x->exp_node = c.take<int>((size_t)B * z.D * z.k);
  const size_t Bk = (size_t)B * z.k;
  x->drow_tok = c.take<int>(Bk); x->drow_pos = c.take<int>(Bk); x->drow_slot = c.take<int>(Bk);
  x->drow_seq = c.take<int>(Bk); x->drow_feat = c.take<int>(Bk); x->drow_plant = c.take<int>(Bk);
  x->drow_out = c.take<int>(Bk); x->dmask = c.take<uint64_t>(Bk * z.dmw);
  const size_t BT = (size_t)B * z.T1;
  x->tree_tok = c.take<int>(BT); x->tree_pos = c.take<int>(BT); x->tree_slot = c.take<int>(BT);
  x->tree_seq = c.take<int>(BT); x->tree_parent = c.take<int>(BT); x->tree_node = c.take<int>(BT);
  x->tree_kids = c.take<int>(BT * z.k); x->tmask = c.take<uint64_t>(BT * z.tmw); x->margin = c.take<float>(BT);
  x->row_tok = c.take<int>(z.R); x->row_pos = c.take<int>(z.R); x->row_slot = c.take<int>(z.R);
  x->row_seq = c.take<int>(z.R); x->row_feat = c.take<int>(z.R);
  const size_t es = z.esz;
  x->x = c.take<float>((size_t)z.R * z.H);
  x->qkv = c.take<float>((size_t)z.R * z.QKV);
  x->gu = c.take<float>((size_t)z.R * 2 * z.F);
  x->ain = c.take<uint8_t>((size_t)z.R * z.KIN * es);
  x->qb = c.take<uint8_t>((size_t)z.R * z.A * es);
  x->att = c.take<uint8_t>((size_t)z.R * z.A * es);
  x->hb = c.take<uint8_t>((size_t)z.R * z.F * es);
  x->feat_t = c.take<uint8_t>((size_t)z.Rt * z.H * es);
  x->caps = c.take<uint8_t>(z.kind == 3 ? (size_t)3 * z.Rt * z.H * es : 16);
  x->dout = c.take<uint8_t>((size_t)z.Rd * z.H * es);
  x->fsrc = c.take<uint8_t>((size_t)B * z.fsrc_rows * z.H * es);
  x->gbuf = c.take<uint8_t>((size_t)z.Rd * z.H * es);
  x->ebuf = c.take<uint8_t>((size_t)z.Rd * z.H * es);
  x->pre_feat = c.take<uint8_t>((size_t)z.max_ctx * z.H * es * (z.kind == 3 ? 3 : 1));
  x->logits = c.take<float>((size_t)z.Rh * z.V);
  x->h_part = c.take<float>(head_part_bytes(z.V, z.Rh, z.Kh) / sizeof(float) + 16);
  x->h_id = c.take<int>((size_t)z.Rh * z.Kh); x->h_val = c.take<float>((size_t)z.Rh * z.Kh);
  x->h_lse = c.take<float>(z.Rh); x->h_spec = c.take<float>((size_t)z.Rh * z.k);
  x->v_id = c.take<int>((size_t)z.B * z.T1 * 2); x->v_val = c.take<float>((size_t)z.B * z.T1 * 2);
  x->v_lse = c.take<float>((size_t)z.B * z.T1); x->v_spec = c.take<float>((size_t)z.B * z.T1 * z.k);
  x->v_logits = c.take<float>((size_t)z.B * z.T1 * z.V);
  x->gemm_part_floats = gemm_bf16_scratch_bytes(std::max(z.R, z.Rh)) / sizeof(float);
  x->gemm_part = c.take<float>(x->gemm_part_floats);
  x->gemm_cnt_len = 65536;
  x->gemm_cnt = c.take<int>(x->gemm_cnt_len);
  {
    // the key splits of the cycle's launches (one per 64-key tile of the larger cache, up to
    // 32); launches with more rows (prefill chunks) run fewer, longer splits in the same space
    // (plus one tail partial per row)
    const int ns = std::max(attention_max_splits(z.cap, z.B), attention_max_splits(z.dcap, z.B)) + 1;
    const int rs = std::max(std::max(std::max(z.B * z.T1, z.B * (z.D + 1)), z.B * z.k) * ns, 2 * z.R);
    x->attn_pfloats = (size_t)rs * z.nq * z.d;
    x->attn_po = c.take<float>(x->attn_pfloats);
    x->attn_pml = c.take<float>((size_t)rs * z.nq * 2);
  }
  x->ttt_tgt = c.take<int>(std::max(z.Rd, z.Rt));
  x->ttt_acc = c.take<float>(4);
  x->ttt_ce = c.take<float>(std::max(z.Rd, z.Rt));
  x->static_exp = c.take<int>(std::max(1, (z.D - 1) * z.k));
  x->static_keep = c.take<int>(z.NG);
  x->kv_table = c.take<int>(std::max(1, z.nblk));
  x->kv_next = c.take<int>(4);
  x->rope_cos = c.take<float>((size_t)z.rope_pos * (z.d / 2));
  x->rope_sin = c.take<float>((size_t)z.rope_pos * (z.d / 2));
  x->kc = c.take<uint8_t>((size_t)z.L * z.kv_layer_elems * es);
  x->vc = c.take<uint8_t>((size_t)z.L * z.kv_layer_elems * es);
  x->page = KvPage{z.kvb_log2 ? x->kv_table : nullptr, z.tab_w, z.kvb_log2};
  x->dkc = c.take<uint8_t>((size_t)B * z.nkv * z.dcap * z.d * es);
  x->dvc = c.take<uint8_t>((size_t)B * z.nkv * z.dcap * z.d * es);
}

int fail(eagle_ctx* c, int code, const std::string& msg) {
  if (c) c->err = msg;
  return code;
}

#define CK(expr)                                                                       \
  do {                                                                                 \
    int _r = (expr);                                                                   \
    if (_r != 0) return fail(ctx, EAGLE_ECUDA, std::string("launch failed: ") + #expr); \
  } while (0)

// ---- building blocks -------------------------------------------------------------------------
int gemm(eagle_ctx* ctx, const void* W, int N, int K, const void* X, int M, int epi, void* out, int ldo,
         const HeadParams* head = nullptr, const QkvEpi* qkv = nullptr) {
  const Dims& z = ctx->z;
  if (z.dt == DT_BF16) {
    const bool prof = ctx->prof_on && 2 * (ctx->prof_n + 1) <= (int)ctx->prof_ev.size();
    if (prof) cudaEventRecord(ctx->prof_ev[2 * ctx->prof_n], ctx->st);
    const int r = gemm_bf16(ctx->st, W, N, K, X, M, epi, out, ldo, ctx->gemm_part, ctx->gemm_part_floats,
                            ctx->gemm_cnt, ctx->gemm_cnt_len, ctx->dev_err, head, true, qkv);
    if (prof) {
      cudaEventRecord(ctx->prof_ev[2 * ctx->prof_n + 1], ctx->st);
      // algorithmic bytes: weight + activation in + output (fp32, bf16, none for the head)
      const bool b16 = epi == EPI_BF16 || epi == EPI_SWIGLU || epi == EPI_QKV;
      const bool paired = epi == EPI_SWIGLU || epi == EPI_GU;
      const double ob = epi == EPI_HEAD ? 0.0
                                        : (double)M * N * (b16 ? 2 : 4) * (epi == EPI_ADD_F32 || epi == EPI_GU ? 2 : 1);
      ctx->prof_bytes[ctx->prof_n] = (double)N * K * 2 * (paired ? 2 : 1) + (double)M * K * 2 + ob;
      ++ctx->prof_n;
    }
    return r;
  }
  return gemm_f32(ctx->st, (const float*)W, N, K, (const float*)X, M, epi, (float*)out, ldo);
}

HeadParams head_params(eagle_ctx* ctx, int rows, int K) {
  HeadParams p{};
  p.vocab = ctx->z.V;
  p.n_rows = rows;
  p.K = K;
  p.inv_t = 1.f;
  p.part = ctx->h_part;
  p.n_tiles = ctx->z.n_tiles;
  p.top_id = ctx->h_id;
  p.top_val = ctx->h_val;
  p.lse = ctx->h_lse;
  p.spec_logit = ctx->h_spec;
  p.seed = ctx->tc.seed;
  p.stream = STREAM_GUMBEL;
  return p;
}

HeadOut head_out(eagle_ctx* ctx, int K, int S) {
  HeadOut h;
  h.top_id = ctx->h_id; h.top_val = ctx->h_val; h.lse = ctx->h_lse; h.spec_logit = ctx->h_spec;
  h.K = K; h.S = S;
  return h;
}

// logits of X rows -> per-row records -> merged top-K / lse.
int lm_head(eagle_ctx* ctx, const void* X, int M, HeadParams& p, float* logits_buf = nullptr,
            bool dump_logits = false) {
  const Dims& z = ctx->z;
  float* lg = logits_buf ? logits_buf : ctx->logits;
  if (z.dt == DT_BF16) {
    CK(gemm(ctx, ctx->w.lm_head, z.V, z.H, X, M, EPI_HEAD, nullptr, 0, &p));
    if (dump_logits) CK(gemm(ctx, ctx->w.lm_head, z.V, z.H, X, M, EPI_F32, lg, z.V));
  } else {
    CK(gemm(ctx, ctx->w.lm_head, z.V, z.H, X, M, EPI_F32, lg, z.V));
    CK(head_partials_from_logits(ctx->st, lg, z.V, p));
  }
  CK(head_merge(ctx->st, p));
  return 0;
}

// Self-attention of one layer over R rows (q in ctx->qb, keys/values already in the cache)
// into ctx->att.
int attend(eagle_ctx* ctx, void* kcache, void* vcache, int cap, int R, int rows_per_seq, const int* slot,
           const int* seq, int mode, int tree_T, const uint64_t* mask, int mask_words, const KvPage& page) {
  const Dims& z = ctx->z;
  AttnArgs a{};
  a.q = ctx->qb; a.kcache = kcache; a.vcache = vcache; a.out = ctx->att;
  a.R = R; a.nq = z.nq; a.nkv = z.nkv; a.d = z.d; a.cap = cap; a.rows_per_seq = rows_per_seq;
  a.row_seq = seq; a.row_slot = slot; a.ctx_len = ctx->ctx_len; a.mode = mode; a.tree_T = tree_T;
  a.mask = mask; a.mask_words = mask_words; a.scale = 1.f / sqrtf((float)z.d);
  a.page = page;
  a.part_o = ctx->attn_po; a.part_ml = ctx->attn_pml; a.part_floats = ctx->attn_pfloats;
  a.err = ctx->dev_err;
  a.max_splits = attention_max_splits(cap, z.B);   // fixed per cache: verify and plain decoding agree
  a.kv_rows = page.table ? (long long)z.nblk * z.nkv << z.kvb_log2 : (long long)z.B * z.nkv * cap;
  a.max_batch = z.B;
  CK(attention(ctx->st, z.dt, a));
  return 0;
}

// One decoder layer over R rows with per-op launches. attn_in: rounded QKV input
// [R][kin]; x: fp32 residual.
int layer_forward(eagle_ctx* ctx, const eagle_layer_weights& lw, int R, const void* attn_in, int kin, void* kcache,
                  void* vcache, int cap, int rows_per_seq, const int* pos, const int* slot, const int* seq, int mode,
                  int tree_T, const uint64_t* mask, int mask_words, const KvPage& page) {
  const Dims& z = ctx->z;
  // the fused epilogue writes a contiguous cache only
  if (z.dt == DT_BF16 && ctx->fuse_epi > 0 && (ctx->fuse_epi & 2) && 128 % z.d == 0 && !page.table) {
    // RoPE, the q output and the KV-cache write in the projection's epilogue
    const QkvEpi q{pos, slot, seq, ctx->rope_cos, ctx->rope_sin, ctx->qb, kcache, vcache, z.nq, z.nkv, z.d, cap};
    CK(gemm(ctx, lw.wqkv, z.QKV, kin, attn_in, R, EPI_QKV, nullptr, 0, nullptr, &q));
  } else {
    CK(gemm(ctx, lw.wqkv, z.QKV, kin, attn_in, R, EPI_F32, ctx->qkv, z.QKV));
    CK(rope_store(ctx->st, z.dt, ctx->qkv, R, z.nq, z.nkv, z.d, pos, slot, seq, ctx->rope_cos, ctx->rope_sin,
                  ctx->qb, kcache, vcache, cap, ctx->dev_err, cap, page));
  }
  int r = attend(ctx, kcache, vcache, cap, R, rows_per_seq, slot, seq, mode, tree_T, mask, mask_words, page);
  if (r) return r;
  CK(gemm(ctx, lw.wo, z.H, z.A, ctx->att, R, EPI_ADD_F32, ctx->x, z.H));
  CK(rmsnorm_rows(ctx->st, DT_F32, ctx->x, z.H, lw.mlp_norm, z.H, ctx->mc.rms_eps, R, z.dt, ctx->ain, z.H));
  // The paired [gate; up] tile layout (64 gate + the matching 64 up features per tile) with
  // SwiGLU in the epilogue, or its fp32 gate/up values and a separate SwiGLU pass (the same
  // bits); the plain layout only for one sequence under EAGLE_FUSE_EPI=-1.
  if (z.dt == DT_BF16 && z.F % 64 == 0 && (ctx->batch > 1 || ctx->fuse_epi >= 0)) {
    if ((ctx->fuse_epi > 0 && (ctx->fuse_epi & 1)) || (ctx->fuse_epi < 0 && R >= 128)) {
      CK(gemm(ctx, lw.wgu, z.F, z.H, ctx->ain, R, EPI_SWIGLU, ctx->hb, z.F));
    } else {
      CK(gemm(ctx, lw.wgu, z.F, z.H, ctx->ain, R, EPI_GU, ctx->gu, 2 * z.F));
      CK(swiglu_rows(ctx->st, z.dt, ctx->gu, z.F, R, ctx->hb));
    }
  } else {
    CK(gemm(ctx, lw.wgu, 2 * z.F, z.H, ctx->ain, R, EPI_F32, ctx->gu, 2 * z.F));
    CK(swiglu_rows(ctx->st, z.dt, ctx->gu, z.F, R, ctx->hb));
  }
  CK(gemm(ctx, lw.wd, z.H, z.F, ctx->hb, R, EPI_ADD_F32, ctx->x, z.H));
  return 0;
}

// Target forward over R rows: features (rounded final-norm output) into feat_out [R][H],
// EAGLE-3 captures into caps_out [3][caps_ld][H] (rows at offset caps_row0).
int target_forward(eagle_ctx* ctx, int R, const int* tok, const int* pos, const int* slot, const int* seq,
                   int rows_per_seq, int mode, int tree_T, const uint64_t* mask, int mask_words, void* feat_out,
                   void* caps_out, size_t caps_ld, size_t caps_row0) {
  const Dims& z = ctx->z;
  CK(embed_rows(ctx->st, z.dt, ctx->w.embed, z.V, z.H, tok, R, ctx->x, ctx->dev_err));
  const size_t lstride = z.kv_layer_elems * z.esz;
  for (int l = 0; l < z.L; ++l) {
    const eagle_layer_weights& lw = ctx->layers[l];
    CK(rmsnorm_rows(ctx->st, DT_F32, ctx->x, z.H, lw.attn_norm, z.H, ctx->mc.rms_eps, R, z.dt, ctx->ain, z.H));
    int r = layer_forward(ctx, lw, R, ctx->ain, z.H, (uint8_t*)ctx->kc + l * lstride, (uint8_t*)ctx->vc + l * lstride,
                          z.cap, rows_per_seq, pos, slot, seq, mode, tree_T, mask, mask_words, ctx->page);
    if (r) return r;
    if (z.kind == 3 && caps_out) {
      for (int j = 0; j < 3; ++j)
        if (ctx->dc.fuse_layers[j] == l)
          CK(convert_rows(ctx->st, z.dt, ctx->x, z.H, R,
                          (uint8_t*)caps_out + ((size_t)j * caps_ld + caps_row0) * z.H * z.esz, z.H));
    }
  }
  CK(rmsnorm_rows(ctx->st, DT_F32, ctx->x, z.H, ctx->w.final_norm, z.H, ctx->mc.rms_eps, R, z.dt, feat_out, z.H));
  return 0;
}

// EAGLE-3: g = FC([l; m; h]) (bf16-rounded) for R rows whose captures are gathered from
// `caps` [3][caps_ld][H] at rows idx (identity if null) -> gbuf [R][H].
int fuse_rows(eagle_ctx* ctx, const void* caps, size_t caps_ld, const int* idx, int R) {
  const Dims& z = ctx->z;
  const size_t rb = (size_t)z.H * z.esz;
  for (int j = 0; j < 3; ++j)
    CK(gather_rows(ctx->st, rb, (const uint8_t*)caps + (size_t)j * caps_ld * rb, rb, idx, R,
                   (uint8_t*)ctx->ain + j * rb, 3 * rb));
  CK(gemm(ctx, ctx->w.fc, z.H, 3 * z.H, ctx->ain, R, z.dt == DT_BF16 ? EPI_BF16 : EPI_F32, ctx->gbuf, z.H));
  return 0;
}

// Drafter step over R rows. Feature input of row r: feat[feat_row[r]] (EAGLE-1: f or the
// parent's predicted feature; EAGLE-3: g or the parent's a). Output (rounded) to ctx->dout.
int drafter_forward(eagle_ctx* ctx, int R, const int* tok, const int* pos, const int* slot, const int* seq,
                    int rows_per_seq, int mode, int tree_T, const uint64_t* mask, int mask_words, const void* feat,
                    const int* feat_row) {
  const Dims& z = ctx->z;
  const eagle_layer_weights& lw = ctx->w.draft;
  const size_t rb = (size_t)z.H * z.esz;
  int kin;
  if (z.kind == 1) {
    CK(concat_emb_feat(ctx->st, z.dt, ctx->w.embed, z.V, z.H, tok, feat, feat_row, R, ctx->ain, ctx->dev_err));
    CK(gemm(ctx, ctx->w.fc, z.H, 2 * z.H, ctx->ain, R, EPI_F32, ctx->x, z.H));
    CK(rmsnorm_rows(ctx->st, DT_F32, ctx->x, z.H, lw.attn_norm, z.H, ctx->mc.rms_eps, R, z.dt, ctx->ain, z.H));
    kin = z.H;
  } else if (z.dt == DT_BF16) {
    CK(eagle3_input_rows(ctx->st, feat, feat_row, ctx->w.embed, z.V, tok, z.H, ctx->w.norm_g, ctx->w.norm_e,
                         ctx->mc.rms_eps, ctx->gbuf, ctx->x, ctx->ebuf, ctx->ain, R, ctx->dev_err));
    kin = 2 * z.H;
  } else {
    if (feat != ctx->gbuf || feat_row)
      CK(gather_rows(ctx->st, rb, feat, rb, feat_row, R, ctx->gbuf, rb));
    CK(widen_rows(ctx->st, z.dt, ctx->gbuf, z.H, z.H, R, ctx->x));
    CK(rmsnorm_rows(ctx->st, z.dt, ctx->gbuf, z.H, ctx->w.norm_g, z.H, ctx->mc.rms_eps, R, z.dt, ctx->ain, 2 * z.H));
    CK(gather_rows(ctx->st, rb, ctx->w.embed, rb, tok, R, ctx->ebuf, rb, nullptr, z.V, ctx->dev_err));
    CK(rmsnorm_rows(ctx->st, z.dt, ctx->ebuf, z.H, ctx->w.norm_e, z.H, ctx->mc.rms_eps, R, z.dt,
                    (uint8_t*)ctx->ain + rb, 2 * z.H));
    kin = 2 * z.H;
  }
  int r = layer_forward(ctx, lw, R, ctx->ain, kin, ctx->dkc, ctx->dvc, z.dcap, rows_per_seq, pos, slot, seq, mode,
                        tree_T, mask, mask_words, KvPage{nullptr, 0, 0});
  if (r) return r;
  CK(convert_rows(ctx->st, z.dt, ctx->x, z.H, R, ctx->dout, z.H));
  return 0;
}

void fill_cd(eagle_ctx* ctx) {
  const Dims& z = ctx->z;
  CycleDev& c = ctx->cd;
  c.B = ctx->batch > 0 ? ctx->batch : z.B;
  c.k = z.k; c.D = z.D; c.m = z.m; c.T1 = z.T1; c.NG = z.NG; c.V = z.V;
  c.kc = ctx->zc.k;
  c.dmask_words = z.dmw; c.tmask_words = z.tmw; c.fsrc_rows = z.fsrc_rows;
  c.ctx_len = ctx->ctx_len; c.n_old = ctx->n_old; c.root_tok = ctx->root_tok; c.committed = ctx->committed;
  c.stop_at = ctx->stop_at;
  c.on_track = ctx->on_track; c.cycle = ctx->cycle;
  c.planted_p = ctx->tc.planted_p; c.planted_conf = ctx->tc.planted_conf;
  c.inv_t = ctx->tc.temperature > 0.f ? 1.f / ctx->tc.temperature : 1.f;
  c.seed = ctx->tc.seed;
  c.sampling = ctx->tc.temperature > 0.f ? 1 : 0;
  c.cand_tok = ctx->cand_tok; c.cand_logc = ctx->cand_logc; c.root_plant = ctx->root_plant;
  c.node_tok = ctx->node_tok; c.node_parent = ctx->node_parent; c.node_depth = ctx->node_depth;
  c.node_logv = ctx->node_logv; c.node_rank = ctx->node_rank; c.exp_node = ctx->exp_node;
  c.drow_tok = ctx->drow_tok; c.drow_pos = ctx->drow_pos; c.drow_slot = ctx->drow_slot; c.drow_seq = ctx->drow_seq;
  c.drow_feat = ctx->drow_feat; c.drow_plant = ctx->drow_plant; c.dmask = ctx->dmask;
  c.tree_tok = ctx->tree_tok; c.tree_pos = ctx->tree_pos; c.tree_slot = ctx->tree_slot; c.tree_seq = ctx->tree_seq;
  c.tree_parent = ctx->tree_parent; c.tree_node = ctx->tree_node; c.tree_kids = ctx->tree_kids; c.tmask = ctx->tmask;
  c.acc_len = ctx->acc_len; c.emitted = ctx->emitted; c.acc_path = ctx->acc_path; c.bonus = ctx->bonus; c.margin = ctx->margin;
  c.err = ctx->dev_err;
  c.policy = ctx->static_on;
  c.static_exp = ctx->static_exp;
  c.static_keep = ctx->static_keep;
}

__global__ void iota_k(int* p, int n) {
  PDL_ENTRY();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) p[i] = i;
}

// rows of the expansion outputs inside the [B][fsrc_rows][H] feature-source buffer
__global__ void drow_out_k(int* out, int B, int k, int fsrc_rows, int d) {
  PDL_ENTRY();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < B * k) out[i] = (i / k) * fsrc_rows + 1 + (d - 1) * k + (i % k);
}

// ---- cycle statistics ---------------------------------------------------------------------------
// The device clock (ns) once the preceding kernel has finished.
__global__ void stamp_k(uint64_t* t) {
  PDL_ENTRY();
  uint64_t ns;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(ns));
  *t = ns;
}

// The batch's totals of the cycle that just ended (one warp, fixed summation order).
__global__ void cycle_stats_k(const int* emitted, const int* acc_len, int B, int m, eagle_cycle_stats* s) {
  PDL_ENTRY();
  int act = 0, acc = 0, emit = 0, mx = 0;
  for (int b = threadIdx.x; b < B; b += 32) {
    const int e = emitted[b], l = e > 0 ? acc_len[b] : 0;
    act += e > 0;
    emit += e;
    acc += l;
    mx = max(mx, l);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    act += __shfl_xor_sync(0xffffffffu, act, off);
    emit += __shfl_xor_sync(0xffffffffu, emit, off);
    acc += __shfl_xor_sync(0xffffffffu, acc, off);
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  }
  if (threadIdx.x == 0) {
    s->batch = B;
    s->active = act;
    s->accepted = acc;
    s->committed = emit;
    s->max_accepted = mx;
    s->verify_rows = m + 1;
  }
}

// ---- paged target KV: block assignment ---------------------------------------------------------
// Every table entry -1 and the pool's counter 0 (at prefill, which starts the sequences anew).
__global__ void kv_reset_k(int* table, int n, int* next) {
  PDL_ENTRY();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) table[i] = -1;
  if (i == 0) *next = 0;
}

// Sequences b0 .. b0 + nb - 1 get pool blocks for their slots [lo, lo + span), lo = lo_dev[b]
// (or lo_const): one thread walks them in order, so placement is deterministic. The pool holds
// every sequence's worst case, so it runs dry only on a host-side capacity bug (latched).
__global__ void kv_reserve_k(int* table, int tab_w, int bs_log2, int* next, int nblk, int b0, int nb,
                             const int* lo_dev, int lo_const, int span, int* err) {
  PDL_ENTRY();
  if (blockIdx.x || threadIdx.x) return;
  int nx = *next;
  for (int b = b0; b < b0 + nb; ++b) {
    const int lo = lo_dev ? lo_dev[b] : lo_const;
    if (span <= 0 || lo < 0) continue;
    const int j0 = lo >> bs_log2, j1 = min((lo + span - 1) >> bs_log2, tab_w - 1);
    for (int j = j0; j <= j1; ++j) {
      int* e = table + (size_t)b * tab_w + j;
      if (*e >= 0) continue;
      if (nx >= nblk) { latch_error(err, DEVERR_CAPACITY); break; }
      *e = nx++;
    }
  }
  *next = nx;
}

int kv_reserve(eagle_ctx* ctx, int b0, int nb, const int* lo_dev, int lo_const, int span) {
  const Dims& z = ctx->z;
  if (!ctx->page.table) return 0;
  launch_k(kv_reserve_k, 1, 32, 0, ctx->st, ctx->kv_table, z.tab_w, z.kvb_log2, ctx->kv_next, z.nblk, b0, nb, lo_dev,
           lo_const, span, ctx->dev_err);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

// ---- training-time-test forward (EAGLE-3 multi-step drafter pass) ------------------------------
// Rows of pass s over a sequence of n tokens: s = 0 the target's causal pass (token x_t at
// position t, slot t); s >= 1 drafter step s, sources t = 0 .. R-1: token x_{t+s} at position
// t+s-1, slot t (s = 1) or n(s-1)+t, target token x_{t+s+1}. The sequence length goes to
// ctx_len[0] (the mode-2 attention reads it).
__global__ void ttt_rows_k(const int* x, int n, int s, int R, int* tok, int* pos, int* slot, int* seq, int* tgt,
                           int* ctx_len) {
  PDL_ENTRY();
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t == 0) ctx_len[0] = n;
  if (t >= R) return;
  if (s == 0) {
    tok[t] = x[t]; pos[t] = t; slot[t] = t; seq[t] = 0;
    return;
  }
  tok[t] = x[t + s];
  pos[t] = t + s - 1;
  slot[t] = s == 1 ? t : n * (s - 1) + t;
  seq[t] = 0;
  tgt[t] = x[t + s + 1];
}

// ce[i] = lse - logit of the target for each row; acc[0] += their sum, in a fixed order;
// one block.
__global__ void ttt_loss_acc_k(const float* lse, const float* tgt_logit, int rows, float* acc, int reset, float* ce) {
  PDL_ENTRY();
  __shared__ float red[256];
  float v = 0.f;
  for (int i = threadIdx.x; i < rows; i += blockDim.x) {
    const float c = lse[i] - tgt_logit[i];
    ce[i] = c;
    v += c;
  }
  red[threadIdx.x] = v;
  __syncthreads();
  for (int o = blockDim.x / 2; o > 0; o >>= 1) {
    if (threadIdx.x < o) red[threadIdx.x] += red[threadIdx.x + o];
    __syncthreads();
  }
  if (threadIdx.x == 0) acc[0] = (reset ? 0.f : acc[0]) + red[0];
}

__global__ void ttt_loss_fin_k(const float* acc, int rows, float* out) {
  PDL_ENTRY();
  if (threadIdx.x == 0 && blockIdx.x == 0) out[0] = acc[0] / (float)rows;
}

// ---- the cycle -------------------------------------------------------------------------------
int enqueue_cycle(eagle_ctx* ctx, int32_t* out_tokens, int32_t* out_count) {
  const Dims& z = ctx->z;
  const int B = ctx->batch;
  CycleDev& c = ctx->cd;
  const size_t rb = (size_t)z.H * z.esz;
  // phase marks: a device clock stamp into the caller's statistics, CUDA events in a profiled
  // window, and an NVTX range around the phase's host-side enqueue
  static const char* const names[PHASES] = {"eagle.draft", "eagle.select", "eagle.verify", "eagle.accept_compact",
                                            "eagle.update"};
  const bool pprof = ctx->prof_on && (size_t)(PHASES + 1) * (ctx->ph_n + 1) <= ctx->ph_ev.size();
  auto mark = [&](int i) {   // i = 0: the cycle's start; i = 1..PHASES: the end of phase i
    if (ctx->stats) launch_k(stamp_k, 1, 32, 0, ctx->st, &ctx->stats->t_ns[i]);
    if (pprof) cudaEventRecord(ctx->ph_ev[(size_t)(PHASES + 1) * ctx->ph_n + i], ctx->st);
    if (i > 0) nvtxRangePop();
    if (i < PHASES) nvtxRangePushA(names[i]);
  };
  mark(0);
  CK(kv_reserve(ctx, 0, B, ctx->ctx_len, 0, z.T1));   // the tree rows' slots [ctx, ctx + m + 1)
  CK(tree_start(ctx->st, c));
  for (int d = 1; d < z.D; ++d) {
    CK(tree_select(ctx->st, c, d));
    int r = drafter_forward(ctx, B * z.k, ctx->drow_tok, ctx->drow_pos, ctx->drow_slot, ctx->drow_seq, z.k, 1, d * z.k,
                            ctx->dmask, z.dmw, ctx->fsrc, ctx->drow_feat);
    if (r) return r;
    if (d + 1 < z.D) {
      launch_k(drow_out_k, (B * z.k + 127) / 128, 128, 0, ctx->st, ctx->drow_out, B, z.k, z.fsrc_rows, d);
      CK(gather_rows(ctx->st, rb, ctx->dout, rb, nullptr, B * z.k, ctx->fsrc, rb, ctx->drow_out));
    }
    HeadParams p = head_params(ctx, B * z.k, z.k);
    p.lse_excl = 1;
    p.specials = ctx->drow_plant;
    p.S = 1;
    r = lm_head(ctx, ctx->dout, B * z.k, p);
    if (r) return r;
    CK(tree_add(ctx->st, c, d, head_out(ctx, z.k, 1)));
  }
  mark(1);
  CK(tree_finalize(ctx->st, c));
  mark(2);
  // verify (target forward over the tree rows, then the LM head epilogue)
  const int RT = B * z.T1;
  int r = target_forward(ctx, RT, ctx->tree_tok, ctx->tree_pos, ctx->tree_slot, ctx->tree_seq, z.T1, 1, z.T1,
                         ctx->tmask, z.tmw, ctx->feat_t, ctx->caps, (size_t)z.Rt, 0);
  if (r) return r;
  const bool sampling = ctx->tc.temperature > 0.f;
  HeadParams p = head_params(ctx, RT, sampling ? 1 : 2);
  if (sampling) {
    p.inv_t = 1.f / ctx->tc.temperature;
    p.gumbel = 1;
    p.specials = ctx->tree_kids;
    p.S = z.k;
    p.row_seq = ctx->tree_seq;
    p.key_mod = z.T1;
    p.cycle = ctx->cycle;
    p.cycle_per_seq = 1;
  }
  p.top_id = ctx->v_id;
  p.top_val = ctx->v_val;
  p.lse = ctx->v_lse;
  p.spec_logit = ctx->v_spec;
  r = lm_head(ctx, ctx->feat_t, RT, p, ctx->v_logits, (ctx->debug & EAGLE_DEBUG_LOGITS) != 0);
  if (r) return r;
  mark(3);
  HeadOut hv;
  hv.top_id = ctx->v_id; hv.top_val = ctx->v_val; hv.lse = ctx->v_lse; hv.spec_logit = ctx->v_spec;
  hv.K = p.K; hv.S = sampling ? z.k : 1;
  CK(accept_walk(ctx->st, c, hv, out_tokens, out_count));
  CK(compact_kv(ctx->st, z.dt, ctx->kc, ctx->vc, z.L, z.kv_layer_elems, z.B, z.nkv, z.cap, z.d, ctx->n_old,
                ctx->acc_len, ctx->acc_path, z.D, ctx->page));
  mark(4);
  // drafter update over the committed positions
  const int RU = B * (z.D + 1);
  CK(update_rows(ctx->st, c, ctx->row_tok, ctx->row_pos, ctx->row_slot, ctx->row_seq, ctx->row_feat));
  if (z.kind == 1) {
    r = drafter_forward(ctx, RU, ctx->row_tok, ctx->row_pos, ctx->row_slot, ctx->row_seq, z.D + 1, 0, 0, nullptr, 0,
                        ctx->feat_t, ctx->row_feat);
  } else {
    r = fuse_rows(ctx, ctx->caps, (size_t)z.Rt, ctx->row_feat, RU);
    if (r) return r;
    r = drafter_forward(ctx, RU, ctx->row_tok, ctx->row_pos, ctx->row_slot, ctx->row_seq, z.D + 1, 0, 0, nullptr, 0,
                        ctx->gbuf, nullptr);
  }
  if (r) return r;
  CK(root_prepare(ctx->st, c, z.D + 1, ctx->root_row));
  // root feature of each sequence -> fsrc row b * fsrc_rows, and the LM-head input rows
  CK(gather_rows(ctx->st, rb, ctx->dout, rb, ctx->root_row, B, ctx->fsrc, (size_t)z.fsrc_rows * rb));
  CK(gather_rows(ctx->st, rb, ctx->dout, rb, ctx->root_row, B, ctx->ebuf, rb));
  HeadParams q = head_params(ctx, B, ctx->zc.k);
  q.lse_excl = 1;
  q.specials = ctx->root_plant;
  q.S = 1;
  r = lm_head(ctx, ctx->ebuf, B, q);
  if (r) return r;
  CK(root_candidates(ctx->st, c, head_out(ctx, ctx->zc.k, 1), 1));
  mark(5);
  if (ctx->stats) launch_k(cycle_stats_k, 1, 32, 0, ctx->st, ctx->emitted, ctx->acc_len, B, z.m, ctx->stats);
  if (pprof) ++ctx->ph_n;
  return cudaGetLastError() == cudaSuccess ? 0 : fail(ctx, EAGLE_ECUDA, "launch failed");
}

// Prefill of B equal-length prompts in one batched pass (rows b * n + p), used when all of
// them fit the activation buffers at once.
int prefill_batched(eagle_ctx* ctx, int B, int n, const int* tokens) {
  const Dims& z = ctx->z;
  CycleDev& c = ctx->cd;
  const size_t rb = (size_t)z.H * z.esz;
  const int R = B * n;
  CK(prefill_rows_batched(ctx->st, tokens, B, n, 0, ctx->root_tok, ctx->row_tok, ctx->row_pos, ctx->row_slot,
                          ctx->row_seq));
  int r = target_forward(ctx, R, ctx->row_tok, ctx->row_pos, ctx->row_slot, ctx->row_seq, n, 0, 0, nullptr, 0,
                         ctx->feat_t, ctx->caps, (size_t)z.Rt, 0);
  if (r) return r;
  // first generated token of every sequence from its last row
  CK(gather_rows(ctx->st, rb, (const uint8_t*)ctx->feat_t + (size_t)(n - 1) * rb, (size_t)n * rb, nullptr, B,
                 ctx->ebuf, rb));
  const bool sampling = ctx->tc.temperature > 0.f;
  HeadParams p = head_params(ctx, B, 1);
  if (sampling) {
    p.inv_t = 1.f / ctx->tc.temperature;
    p.gumbel = 1;
    p.row_seq = ctx->iota;
    p.key_mod = 1;
    p.cycle_const = PREFILL_CYCLE;
  }
  r = lm_head(ctx, ctx->ebuf, B, p);
  if (r) return r;
  CK(prefill_finish_batched(ctx->st, c, n, ctx->h_id, 1));
  // drafter over the prompt positions (token advanced by one step)
  CK(prefill_rows_batched(ctx->st, tokens, B, n, 1, ctx->root_tok, ctx->row_tok, ctx->row_pos, ctx->row_slot,
                          ctx->row_seq));
  if (z.kind == 1) {
    r = drafter_forward(ctx, R, ctx->row_tok, ctx->row_pos, ctx->row_slot, ctx->row_seq, n, 0, 0, nullptr, 0,
                        ctx->feat_t, ctx->iota);
  } else {
    r = fuse_rows(ctx, ctx->caps, (size_t)z.Rt, nullptr, R);
    if (r) return r;
    r = drafter_forward(ctx, R, ctx->row_tok, ctx->row_pos, ctx->row_slot, ctx->row_seq, n, 0, 0, nullptr, 0,
                        ctx->gbuf, nullptr);
  }
  if (r) return r;
  const uint8_t* last = (const uint8_t*)ctx->dout + (size_t)(n - 1) * rb;
  CK(gather_rows(ctx->st, rb, last, (size_t)n * rb, nullptr, B, ctx->fsrc, (size_t)z.fsrc_rows * rb));
  CK(gather_rows(ctx->st, rb, last, (size_t)n * rb, nullptr, B, ctx->ebuf, rb));
  HeadParams q = head_params(ctx, B, ctx->zc.k);
  q.lse_excl = 1;
  q.specials = ctx->root_plant;
  q.S = 1;
  r = lm_head(ctx, ctx->ebuf, B, q);
  if (r) return r;
  CK(root_candidates(ctx->st, c, head_out(ctx, ctx->zc.k, 1), 0));
  return 0;
}

// No sequence has a limit (a fresh batch of sequences starts unlimited).
int clear_stops(eagle_ctx* ctx) {
  std::vector<int> none(ctx->z.B, INT32_MAX);
  return cudaMemcpyAsync(ctx->stop_at, none.data(), none.size() * sizeof(int), cudaMemcpyHostToDevice, ctx->st) ==
                 cudaSuccess
             ? 0
             : -4;
}

int check_dev_error(eagle_ctx* ctx) {
  int h[4] = {0, 0, 0, 0};
  std::vector<int> lens(ctx->batch > 0 ? ctx->batch : 1, 0);
  if (cudaMemcpyAsync(h, ctx->dev_err, sizeof(h), cudaMemcpyDeviceToHost, ctx->st) != cudaSuccess ||
      cudaMemcpyAsync(lens.data(), ctx->ctx_len, lens.size() * sizeof(int), cudaMemcpyDeviceToHost, ctx->st) !=
          cudaSuccess)
    return fail(ctx, EAGLE_ECUDA, "reading the device status word failed");
  if (cudaStreamSynchronize(ctx->st) != cudaSuccess)
    return fail(ctx, EAGLE_ECUDA, std::string("stream error: ") + cudaGetErrorString(cudaGetLastError()));
  // the exact lengths replace the host's worst-case bound
  long long mx = 0;
  for (int v : lens) mx = std::max<long long>(mx, v);
  ctx->host_ctx_bound = mx;
  if (h[0]) {
    cudaMemsetAsync(ctx->dev_err, 0, sizeof(int) * 4, ctx->st);
    cudaStreamSynchronize(ctx->st);
    switch (h[0]) {
      case DEVERR_MBAR_TIMEOUT: return fail(ctx, EAGLE_ETIMEOUT, "a device wait exceeded its time limit");
      case DEVERR_CAPACITY: return fail(ctx, EAGLE_EDEVICE, "a KV slot beyond the cache capacity was requested");
      default: return fail(ctx, EAGLE_EDEVICE, "a device-side bounds check failed");
    }
  }
  return EAGLE_OK;
}

}  // namespace

// ---- C ABI ---------------------------------------------------------------------------------------
extern "C" {

size_t eagle_workspace_bytes(const eagle_model_cfg* model, const eagle_drafter_cfg* drafter, const eagle_tree_cfg* tree,
                             const eagle_limits* limits) {
  Dims z;
  std::string why;
  if (!derive(model, drafter, tree, limits, z, why)) return 0;
  eagle_ctx tmp;
  Carver c;
  carve(c, &tmp, z);
  return align_up(c.off, 256) + 256;
}

int eagle_create(const eagle_model_cfg* model, const eagle_drafter_cfg* drafter, const eagle_tree_cfg* tree,
                 const eagle_weights* weights, const eagle_limits* limits, void* workspace, size_t ws_bytes,
                 void* stream, eagle_ctx** out) {
  if (!out) return EAGLE_EINVAL;
  *out = nullptr;
  Dims z;
  std::string why;
  if (!derive(model, drafter, tree, limits, z, why)) {
    fprintf(stderr, "eagle_create: %s\n", why.c_str());
    return EAGLE_EINVAL;
  }
  if (!weights || !weights->embed || !weights->lm_head || !weights->final_norm || !weights->layers || !weights->fc ||
      !weights->draft.wqkv || !weights->draft.wo || !weights->draft.mlp_norm || !weights->draft.wgu ||
      !weights->draft.wd || (drafter->kind == 1 && !weights->draft.attn_norm) ||
      (drafter->kind == 3 && (!weights->norm_g || !weights->norm_e))) {
    fprintf(stderr, "eagle_create: missing weight pointer\n");
    return EAGLE_EINVAL;
  }
  for (int l = 0; l < model->n_layers; ++l) {
    const eagle_layer_weights& lw = weights->layers[l];
    if (!lw.attn_norm || !lw.wqkv || !lw.wo || !lw.mlp_norm || !lw.wgu || !lw.wd) {
      fprintf(stderr, "eagle_create: missing weight pointer in layer %d\n", l);
      return EAGLE_EINVAL;
    }
  }
  if (!workspace) return EAGLE_EINVAL;
  const size_t need = eagle_workspace_bytes(model, drafter, tree, limits);
  if (ws_bytes < need) {
    fprintf(stderr, "eagle_create: workspace of %zu bytes is smaller than the %zu required\n", ws_bytes, need);
    return EAGLE_ECAPACITY;
  }
  if (getenv("EAGLE_FAULT") && strcmp(getenv("EAGLE_FAULT"), "create") == 0) return EAGLE_ECUDA;
  eagle_ctx* ctx = new eagle_ctx();
  ctx->z = z;
  ctx->zc = z;
  ctx->mc = *model; ctx->dc = *drafter; ctx->tc = *tree; ctx->lim = *limits;
  ctx->w = *weights;
  ctx->layers.assign(weights->layers, weights->layers + model->n_layers);
  ctx->w.layers = ctx->layers.data();
  ctx->st = reinterpret_cast<cudaStream_t>(stream);
  if (getenv("EAGLE_FUSE_EPI")) ctx->fuse_epi = atoi(getenv("EAGLE_FUSE_EPI")) & 3;
  Carver c;
  c.base = reinterpret_cast<uint8_t*>(align_up(reinterpret_cast<uintptr_t>(workspace), 256));
  carve(c, ctx, z);
  // zero the state and scratch (tickets must start at zero); the KV caches need no init
  const size_t state_bytes = (uint8_t*)ctx->kc - c.base;
  if (cudaMemsetAsync(c.base, 0, state_bytes, ctx->st) != cudaSuccess) { delete ctx; return EAGLE_ECUDA; }
  // rotary tables in double precision on the host
  const int half = z.d / 2;
  std::vector<float> cs((size_t)z.rope_pos * half), sn((size_t)z.rope_pos * half);
  for (int p = 0; p < z.rope_pos; ++p)
    for (int i = 0; i < half; ++i) {
      const double inv = std::pow((double)model->rope_theta, -2.0 * i / z.d);
      const double a = (double)p * inv;
      cs[(size_t)p * half + i] = (float)std::cos(a);
      sn[(size_t)p * half + i] = (float)std::sin(a);
    }
  if (cudaMemcpyAsync(ctx->rope_cos, cs.data(), cs.size() * 4, cudaMemcpyHostToDevice, ctx->st) != cudaSuccess ||
      cudaMemcpyAsync(ctx->rope_sin, sn.data(), sn.size() * 4, cudaMemcpyHostToDevice, ctx->st) != cudaSuccess) {
    delete ctx;
    return EAGLE_ECUDA;
  }
  launch_k(iota_k, (std::max(z.B, z.R) + 127) / 128, 128, 0, ctx->st, ctx->iota, std::max(z.B, z.R));
  if (clear_stops(ctx)) { delete ctx; return EAGLE_ECUDA; }
  if (ctx->page.table)   // no blocks assigned yet (zero would name block 0)
    launch_k(kv_reset_k, (z.nblk + 255) / 256, 256, 0, ctx->st, ctx->kv_table, z.nblk, ctx->kv_next);
  if (cudaStreamSynchronize(ctx->st) != cudaSuccess) { delete ctx; return EAGLE_ECUDA; }
  ctx->batch = z.B;
  fill_cd(ctx);
  *out = ctx;
  return EAGLE_OK;
}

int eagle_prefill(eagle_ctx* ctx, int batch, const int32_t* d_tokens, const int32_t* h_lens, const int32_t* d_ref,
                  int ref_len) {
  if (!ctx) return EAGLE_EINVAL;
  const Dims& z = ctx->z;
  if (batch < 1 || batch > z.B || !d_tokens || !h_lens) return fail(ctx, EAGLE_EINVAL, "bad prefill arguments");
  if (d_ref && ref_len < 2) return fail(ctx, EAGLE_EINVAL, "ref_len must be >= 2");
  long long mx = 0;
  for (int b = 0; b < batch; ++b) {
    if (h_lens[b] < 1) return fail(ctx, EAGLE_EINVAL, "prompt lengths must be >= 1");
    mx = std::max<long long>(mx, h_lens[b]);
  }
  if (mx + z.D + 1 > z.max_ctx) return fail(ctx, EAGLE_ECAPACITY, "prompt longer than max_ctx allows");
  if (getenv("EAGLE_FAULT") && strcmp(getenv("EAGLE_FAULT"), "prefill") == 0)
    return fail(ctx, EAGLE_ECUDA, "injected prefill fault");
  // the captured cycle bakes in the batch size and the reference pointer
  if (ctx->graph && (ctx->graph_batch != batch || ctx->graph_ref != d_ref || ctx->ref_len != (d_ref ? ref_len : 0))) {
    cudaGraphExecDestroy(ctx->graph);
    ctx->graph = nullptr;
  }
  ctx->batch = batch;
  ctx->ref_len = d_ref ? ref_len : 0;
  fill_cd(ctx);
  ctx->cd.ref = d_ref;
  ctx->cd.ref_len = ctx->ref_len;
  CycleDev& c = ctx->cd;
  CK(clear_stops(ctx));
  if (ctx->page.table) {
    // the sequences start anew: empty block table, then blocks for every prompt slot
    launch_k(kv_reset_k, (z.nblk + 255) / 256, 256, 0, ctx->st, ctx->kv_table, z.nblk, ctx->kv_next);
    if (cudaGetLastError() != cudaSuccess) return fail(ctx, EAGLE_ECUDA, "kv table reset failed");
    for (int b = 0; b < batch; ++b) CK(kv_reserve(ctx, b, 1, nullptr, 0, h_lens[b]));
  }
  const size_t rb = (size_t)z.H * z.esz;
  bool uniform = true;
  for (int b = 1; b < batch; ++b) uniform = uniform && h_lens[b] == h_lens[0];
  if (batch > 1 && uniform && (long long)batch * h_lens[0] <= std::min(z.Rt, z.Rd)) {
    const int r = prefill_batched(ctx, batch, h_lens[0], d_tokens);
    if (r) return r;
    ctx->host_ctx_bound = mx;
    return EAGLE_OK;
  }
  long long off = 0;
  for (int b = 0; b < batch; ++b) {
    const int n = h_lens[b];
    const int* prompt = d_tokens + off;
    // target over the prompt in chunks (causal)
    for (int p0 = 0; p0 < n; p0 += z.P) {
      const int R = std::min(z.P, n - p0);
      CK(prefill_rows(ctx->st, prompt, b, p0, R, n, ctx->root_tok, ctx->row_tok, ctx->row_pos, ctx->row_slot,
                      ctx->row_seq, 0));
      int r = target_forward(ctx, R, ctx->row_tok, ctx->row_pos, ctx->row_slot, ctx->row_seq, R, 0, 0, nullptr, 0,
                             ctx->feat_t, ctx->pre_feat, (size_t)z.max_ctx, (size_t)p0);
      if (r) return r;
      if (z.kind == 1)
        CK(gather_rows(ctx->st, (size_t)R * rb, ctx->feat_t, 0, nullptr, 1, (uint8_t*)ctx->pre_feat + (size_t)p0 * rb, 0));
      if (p0 + R == n) {
        // first generated token from the last row
        const bool sampling = ctx->tc.temperature > 0.f;
        HeadParams p = head_params(ctx, 1, 1);
        if (sampling) {
          p.inv_t = 1.f / ctx->tc.temperature;
          p.gumbel = 1;
          p.seq_base = b;
          p.key_mod = 1;
          p.cycle_const = PREFILL_CYCLE;
        }
        r = lm_head(ctx, (uint8_t*)ctx->feat_t + (size_t)(R - 1) * rb, 1, p);
        if (r) return r;
        CK(prefill_finish(ctx->st, c, b, n, ctx->h_id));
      }
    }
    // drafter over positions 0..n-1 (token advanced by one step)
    for (int p0 = 0; p0 < n; p0 += z.P) {
      const int R = std::min(z.P, n - p0);
      CK(prefill_rows(ctx->st, prompt, b, p0, R, n, ctx->root_tok, ctx->row_tok, ctx->row_pos, ctx->row_slot,
                      ctx->row_seq, 1));
      int r;
      if (z.kind == 1) {
        r = drafter_forward(ctx, R, ctx->row_tok, ctx->row_pos, ctx->row_slot, ctx->row_seq, R, 0, 0, nullptr, 0,
                            (uint8_t*)ctx->pre_feat + (size_t)p0 * rb, ctx->iota);
      } else {
        r = fuse_rows(ctx, (uint8_t*)ctx->pre_feat + (size_t)p0 * rb, (size_t)z.max_ctx, nullptr, R);
        if (r) return r;
        r = drafter_forward(ctx, R, ctx->row_tok, ctx->row_pos, ctx->row_slot, ctx->row_seq, R, 0, 0, nullptr, 0,
                            ctx->gbuf, nullptr);
      }
      if (r) return r;
      if (p0 + R == n) {
        const uint8_t* last = (const uint8_t*)ctx->dout + (size_t)(R - 1) * rb;
        CK(gather_rows(ctx->st, rb, last, rb, nullptr, 1, (uint8_t*)ctx->fsrc + (size_t)b * z.fsrc_rows * rb, rb));
        CK(gather_rows(ctx->st, rb, last, rb, nullptr, 1, ctx->ebuf, rb));
        HeadParams q = head_params(ctx, 1, ctx->zc.k);
        q.lse_excl = 1;
        q.specials = ctx->root_plant + b;
        q.S = 1;
        r = lm_head(ctx, ctx->ebuf, 1, q);
        if (r) return r;
        CK(root_candidates_seq(ctx->st, c, head_out(ctx, ctx->zc.k, 1), b));
      }
    }
    off += n;
  }
  ctx->host_ctx_bound = mx;
  return EAGLE_OK;
}

static int run_cycle(eagle_ctx* ctx, int32_t* d_out_tokens, int32_t* d_out_count, eagle_cycle_stats* d_stats);

int eagle_cycle(eagle_ctx* ctx, int32_t* d_out_tokens, int32_t* d_out_count, eagle_cycle_stats* d_stats) {
  if (!ctx) return EAGLE_EINVAL;
  if (d_stats && (reinterpret_cast<uintptr_t>(d_stats) & 7))
    return fail(ctx, EAGLE_EINVAL, "d_stats must be 8-byte aligned");
  const Dims& z = ctx->z;
  if (ctx->host_ctx_bound + z.D + 1 > z.max_ctx)
    return fail(ctx, EAGLE_ECAPACITY, "a sequence could outgrow max_ctx in this cycle");
  if (getenv("EAGLE_FAULT") && strcmp(getenv("EAGLE_FAULT"), "cycle") == 0)
    return fail(ctx, EAGLE_ECUDA, "injected cycle fault");
  ctx->host_ctx_bound += z.D + 1;
  ctx->stats = d_stats;
  nvtxRangePushA("eagle.cycle");
  const int rc = run_cycle(ctx, d_out_tokens, d_out_count, d_stats);
  nvtxRangePop();
  return rc;
}

static int run_cycle(eagle_ctx* ctx, int32_t* d_out_tokens, int32_t* d_out_count, eagle_cycle_stats* d_stats) {
  if (ctx->graph_enabled) {
    if (ctx->graph && (ctx->graph_out != d_out_tokens || ctx->graph_cnt != d_out_count || ctx->graph_stats != d_stats)) {
      cudaGraphExecDestroy(ctx->graph);
      ctx->graph = nullptr;
    }
    if (!ctx->graph) {
      cudaGraph_t g;
      if (cudaStreamBeginCapture(ctx->st, cudaStreamCaptureModeThreadLocal) != cudaSuccess)
        return fail(ctx, EAGLE_ECUDA, "stream capture could not start (graph mode needs a non-default stream)");
      int r = enqueue_cycle(ctx, d_out_tokens, d_out_count);
      cudaError_t e = cudaStreamEndCapture(ctx->st, &g);
      if (r) return r;
      if (e != cudaSuccess) return fail(ctx, EAGLE_ECUDA, "stream capture failed");
      size_t nn = 0;
      cudaGraphGetNodes(g, nullptr, &nn);
      std::vector<cudaGraphNode_t> nodes(nn);
      if (nn) cudaGraphGetNodes(g, nodes.data(), &nn);
      int kn = 0;
      for (auto n : nodes) {
        cudaGraphNodeType ty;
        if (cudaGraphNodeGetType(n, &ty) == cudaSuccess && ty == cudaGraphNodeTypeKernel) ++kn;
      }
      e = cudaGraphInstantiate(&ctx->graph, g, 0);
      cudaGraphDestroy(g);
      if (e != cudaSuccess) { ctx->graph = nullptr; return fail(ctx, EAGLE_ECUDA, "graph instantiation failed"); }
      ctx->graph_out = d_out_tokens;
      ctx->graph_cnt = d_out_count;
      ctx->graph_stats = d_stats;
      ctx->graph_ref = ctx->cd.ref;
      ctx->graph_batch = ctx->batch;
      ctx->graph_kernels = kn;
    }
    if (cudaGraphLaunch(ctx->graph, ctx->st) != cudaSuccess) return fail(ctx, EAGLE_ECUDA, "graph launch failed");
    return EAGLE_OK;
  }
  return enqueue_cycle(ctx, d_out_tokens, d_out_count);
}

int eagle_decode_plain(eagle_ctx* ctx, int n_steps, int32_t* d_out_tokens, float* d_out_margin) {
  if (!ctx) return EAGLE_EINVAL;
  const Dims& z = ctx->z;
  if (n_steps < 0) return fail(ctx, EAGLE_EINVAL, "n_steps must be >= 0");
  if (ctx->host_ctx_bound + n_steps > z.max_ctx) return fail(ctx, EAGLE_ECAPACITY, "plain decoding would outgrow max_ctx");
  const int B = ctx->batch;
  CycleDev& c = ctx->cd;
  const bool sampling = ctx->tc.temperature > 0.f;
  for (int s = 0; s < n_steps; ++s) {
    CK(kv_reserve(ctx, 0, B, ctx->ctx_len, 0, 1));
    CK(plain_rows(ctx->st, c, ctx->row_tok, ctx->row_pos, ctx->row_slot, ctx->row_seq));
    int r = target_forward(ctx, B, ctx->row_tok, ctx->row_pos, ctx->row_slot, ctx->row_seq, 1, 0, 0, nullptr, 0,
                           ctx->feat_t, nullptr, 0, 0);
    if (r) return r;
    // greedy keeps the top two (argmax and the top-2 margin); sampling keeps the Gumbel-argmax
    HeadParams p = head_params(ctx, B, sampling ? 1 : 2);
    if (sampling) {
      p.inv_t = 1.f / ctx->tc.temperature;
      p.gumbel = 1;
      p.row_seq = ctx->iota;
      p.key_mod = 1;
      p.cycle_const = (uint32_t)s;
      p.stream = STREAM_PLAIN;
    }
    r = lm_head(ctx, ctx->feat_t, B, p);
    if (r) return r;
    CK(plain_advance(ctx->st, c, ctx->h_id, p.K, ctx->h_val, d_out_tokens, d_out_margin, n_steps, s));
  }
  ctx->host_ctx_bound += n_steps;
  return EAGLE_OK;
}

int eagle_set_stop(eagle_ctx* ctx, int n, const int32_t* h_limits) {
  if (!ctx) return EAGLE_EINVAL;
  if (n == 0) {
    CK(clear_stops(ctx));
    return EAGLE_OK;
  }
  if (n != ctx->batch || !h_limits) return fail(ctx, EAGLE_EINVAL, "one limit per sequence of the batch");
  std::vector<int> lim(ctx->z.B, INT32_MAX);
  for (int b = 0; b < n; ++b) {
    if (h_limits[b] < 1) return fail(ctx, EAGLE_EINVAL, "limits must be >= 1 committed token");
    lim[b] = h_limits[b];
  }
  if (cudaMemcpyAsync(ctx->stop_at, lim.data(), lim.size() * sizeof(int), cudaMemcpyHostToDevice, ctx->st) !=
          cudaSuccess ||
      cudaStreamSynchronize(ctx->st) != cudaSuccess)
    return fail(ctx, EAGLE_ECUDA, "limit upload failed");
  return EAGLE_OK;
}

int eagle_set_tree_budget(eagle_ctx* ctx, int topk, int m) {
  if (!ctx) return EAGLE_EINVAL;
  const Dims& zc = ctx->zc;
  Dims& z = ctx->z;
  const int NG = topk + (z.D - 1) * topk * topk;
  if (topk < 1 || topk > zc.k || m < 1 || m > zc.m || m > NG)
    return fail(ctx, EAGLE_EINVAL, "topk and m must be at most the values the context was created with");
  if (ctx->static_on) return fail(ctx, EAGLE_EINVAL, "a static tree is set: remove it first");
  z.k = topk;
  z.m = m;
  z.T1 = m + 1;
  z.NG = NG;
  z.dmw = std::max(1, ((z.D - 1) * topk + 63) / 64);
  z.tmw = (z.T1 + 63) / 64;
  z.Kh = std::max(topk, 2);
  ctx->tc.topk = topk;
  ctx->tc.m = m;
  const int32_t* ref = ctx->cd.ref;
  const int ref_len = ctx->cd.ref_len;
  fill_cd(ctx);
  ctx->cd.ref = ref;
  ctx->cd.ref_len = ref_len;
  if (ctx->graph) { cudaGraphExecDestroy(ctx->graph); ctx->graph = nullptr; }   // the sizes are kernel arguments
  return EAGLE_OK;
}

int eagle_cycle_kernel_launches(const eagle_ctx* ctx) { return ctx ? ctx->graph_kernels : -1; }

int eagle_set_graph(eagle_ctx* ctx, int enable) {
  if (!ctx) return EAGLE_EINVAL;
  ctx->graph_enabled = enable ? 1 : 0;
  if (!enable && ctx->graph) { cudaGraphExecDestroy(ctx->graph); ctx->graph = nullptr; }
  return EAGLE_OK;
}

int eagle_profile_begin(eagle_ctx* ctx, int max_launches) {
  if (!ctx || max_launches < 0) return EAGLE_EINVAL;
  if (ctx->graph_enabled) return fail(ctx, EAGLE_EINVAL, "GEMM profiling runs with graph replay off");
  for (auto e : ctx->prof_ev) cudaEventDestroy(e);
  ctx->prof_ev.assign(2 * (size_t)max_launches, nullptr);
  for (auto& e : ctx->prof_ev)
    if (cudaEventCreate(&e) != cudaSuccess) return fail(ctx, EAGLE_ECUDA, "event creation failed");
  ctx->prof_bytes.assign(max_launches, 0.0);
  ctx->prof_n = 0;
  for (auto e : ctx->ph_ev) cudaEventDestroy(e);
  ctx->ph_ev.assign((size_t)(PHASES + 1) * 64, nullptr);
  for (auto& e : ctx->ph_ev)
    if (cudaEventCreate(&e) != cudaSuccess) return fail(ctx, EAGLE_ECUDA, "event creation failed");
  ctx->ph_n = 0;
  ctx->ph_done = 0;
  for (double& t : ctx->ph_ms) t = 0.0;
  ctx->prof_on = 1;
  return EAGLE_OK;
}

int eagle_profile_end(eagle_ctx* ctx, int* launches, double* total_ms, double* total_bytes) {
  if (!ctx || !ctx->prof_on) return EAGLE_EINVAL;
  ctx->prof_on = 0;
  if (cudaStreamSynchronize(ctx->st) != cudaSuccess) return fail(ctx, EAGLE_ECUDA, "stream error");
  double ms = 0, bytes = 0;
  for (int i = 0; i < ctx->prof_n; ++i) {
    float t = 0.f;
    if (cudaEventElapsedTime(&t, ctx->prof_ev[2 * i], ctx->prof_ev[2 * i + 1]) != cudaSuccess)
      return fail(ctx, EAGLE_ECUDA, "event timing failed");
    ms += t;
    bytes += ctx->prof_bytes[i];
  }
  if (launches) *launches = ctx->prof_n;
  if (total_ms) *total_ms = ms;
  if (total_bytes) *total_bytes = bytes;
  for (auto e : ctx->prof_ev) cudaEventDestroy(e);
  ctx->prof_ev.clear();
  for (int p = 0; p < PHASES; ++p) ctx->ph_ms[p] = 0.0;
  for (int i = 0; i < ctx->ph_n; ++i)
    for (int p = 0; p < PHASES; ++p) {
      float t = 0.f;
      const size_t e = (size_t)(PHASES + 1) * i + p;
      if (cudaEventElapsedTime(&t, ctx->ph_ev[e], ctx->ph_ev[e + 1]) != cudaSuccess)
        return fail(ctx, EAGLE_ECUDA, "event timing failed");
      ctx->ph_ms[p] += t;
    }
  ctx->ph_done = ctx->ph_n;
  for (auto e : ctx->ph_ev) cudaEventDestroy(e);
  ctx->ph_ev.clear();
  return EAGLE_OK;
}

int eagle_profile_verify(const eagle_ctx* ctx, int* passes, double* total_ms) {
  if (!ctx) return EAGLE_EINVAL;
  if (passes) *passes = ctx->ph_done;
  if (total_ms) *total_ms = ctx->ph_ms[2];
  return EAGLE_OK;
}

int eagle_profile_phases(const eagle_ctx* ctx, int* cycles, double* phase_ms) {
  if (!ctx) return EAGLE_EINVAL;
  if (cycles) *cycles = ctx->ph_done;
  if (phase_ms)
    for (int p = 0; p < PHASES; ++p) phase_ms[p] = ctx->ph_ms[p];
  return EAGLE_OK;
}

int eagle_set_debug(eagle_ctx* ctx, int flags) {
  if (!ctx) return EAGLE_EINVAL;
  ctx->debug = flags;
  if (ctx->graph) { cudaGraphExecDestroy(ctx->graph); ctx->graph = nullptr; }
  return EAGLE_OK;
}

int eagle_status_sync(eagle_ctx* ctx) {
  if (!ctx) return EAGLE_EINVAL;
  return check_dev_error(ctx);
}

size_t eagle_dump_bytes(const eagle_ctx* ctx, int what) {
  if (!ctx) return 0;
  const Dims& z = ctx->z;
  const size_t B = ctx->batch;
  switch (what) {
    case EAGLE_DUMP_STATE: return 7 * B * 4;
    case EAGLE_DUMP_CAND: return 2 * B * ctx->zc.k * 4;
    case EAGLE_DUMP_NODES: return 4 * B * z.NG * 4;
    case EAGLE_DUMP_TREE: return 4 * B * z.T1 * 4 + B * z.T1 * z.tmw * 8;
    case EAGLE_DUMP_ACCEPT: return (2 * B + B * z.D) * 4;
    case EAGLE_DUMP_VERIFY_HEAD: {
      const size_t K = ctx->tc.temperature > 0.f ? 1 : 2;
      const size_t R = B * z.T1;
      return R * K * 8 + R * 4 + R * z.k * 4;
    }
    case EAGLE_DUMP_VERIFY_LOGITS: return B * z.T1 * (size_t)z.V * 4;
    case EAGLE_DUMP_FEATURES: return B * z.T1 * (size_t)z.H * z.esz;
    case EAGLE_DUMP_TTT: return (size_t)ctx->ttt_rows * ((size_t)z.H * z.esz + 4);
  }
  return 0;
}

int eagle_debug_dump(eagle_ctx* ctx, int what, void* dst, size_t bytes) {
  if (!ctx || !dst) return EAGLE_EINVAL;
  const size_t need = eagle_dump_bytes(ctx, what);
  if (!need || bytes < need) return fail(ctx, EAGLE_EINVAL, "dump buffer too small or unknown view");
  const Dims& z = ctx->z;
  const size_t B = ctx->batch;
  uint8_t* o = reinterpret_cast<uint8_t*>(dst);
  auto cp = [&](const void* src, size_t n) {
    cudaMemcpyAsync(o, src, n, cudaMemcpyDeviceToDevice, ctx->st);
    o += n;
  };
  switch (what) {
    case EAGLE_DUMP_STATE:
      cp(ctx->ctx_len, B * 4); cp(ctx->root_tok, B * 4); cp(ctx->committed, B * 4); cp(ctx->on_track, B * 4);
      cp(ctx->cycle, B * 4); cp(ctx->acc_len, B * 4); cp(ctx->bonus, B * 4);
      break;
    case EAGLE_DUMP_CAND: cp(ctx->cand_tok, B * ctx->zc.k * 4); cp(ctx->cand_logc, B * ctx->zc.k * 4); break;
    case EAGLE_DUMP_NODES:
      cp(ctx->node_tok, B * z.NG * 4); cp(ctx->node_parent, B * z.NG * 4); cp(ctx->node_depth, B * z.NG * 4);
      cp(ctx->node_logv, B * z.NG * 4);
      break;
    case EAGLE_DUMP_TREE:
      cp(ctx->tree_tok, B * z.T1 * 4); cp(ctx->tree_pos, B * z.T1 * 4); cp(ctx->tree_parent, B * z.T1 * 4);
      cp(ctx->tree_node, B * z.T1 * 4); cp(ctx->tmask, B * z.T1 * z.tmw * 8);
      break;
    case EAGLE_DUMP_ACCEPT: cp(ctx->acc_len, B * 4); cp(ctx->bonus, B * 4); cp(ctx->acc_path, B * z.D * 4); break;
    case EAGLE_DUMP_VERIFY_HEAD: {
      const size_t K = ctx->tc.temperature > 0.f ? 1 : 2;
      const size_t R = B * z.T1;
      cp(ctx->v_id, R * K * 4); cp(ctx->v_val, R * K * 4); cp(ctx->v_lse, R * 4); cp(ctx->v_spec, R * z.k * 4);
      break;
    }
    case EAGLE_DUMP_VERIFY_LOGITS: cp(ctx->v_logits, B * z.T1 * (size_t)z.V * 4); break;
    case EAGLE_DUMP_FEATURES: cp(ctx->feat_t, B * z.T1 * (size_t)z.H * z.esz); break;
    case EAGLE_DUMP_TTT:
      cp(ctx->dout, (size_t)ctx->ttt_rows * z.H * z.esz);
      cp(ctx->ttt_ce, (size_t)ctx->ttt_rows * 4);
      break;
  }
  return cudaGetLastError() == cudaSuccess ? EAGLE_OK : fail(ctx, EAGLE_ECUDA, "dump copy failed");
}

int eagle_kv_view(const eagle_ctx* ctx, void** k, void** v, int* cap) {
  if (!ctx) return EAGLE_EINVAL;
  if (k) *k = ctx->kc;
  if (v) *v = ctx->vc;
  if (cap) *cap = ctx->z.cap;
  return EAGLE_OK;
}

// Static (EAGLE-1) tree: node i = (parent[i], rank[i]), parent -1 = the root, rank r = the
// drafter's r-th best child. Generation indices follow the drafter's order (depth-1 nodes
// 0..k-1 by rank; the children of the r-th row expanded at depth d start at
// k + (d-1) k^2 + r k); the k rows expanded at depth d are the topology's nodes with
// children in topology order, then the lowest-index other nodes of that depth.
int eagle_set_static_tree(eagle_ctx* ctx, int n, const int32_t* parent, const int32_t* rank) {
  if (!ctx) return EAGLE_EINVAL;
  const Dims& z = ctx->z;
  if (n == 0) {
    ctx->static_on = 0;
  } else {
    if (n != z.m || !parent || !rank) return fail(ctx, EAGLE_EINVAL, "a static tree needs m nodes (parent, rank)");
    std::vector<int> dep(n), gen(n, -1), cnt_exp(z.D + 1, 0);
    for (int i = 0; i < n; ++i) {
      if (parent[i] >= i || parent[i] < -1) return fail(ctx, EAGLE_EINVAL, "parents must precede their children");
      if (rank[i] < 0 || rank[i] >= z.k) return fail(ctx, EAGLE_EINVAL, "rank out of range");
      dep[i] = parent[i] < 0 ? 1 : dep[parent[i]] + 1;
      if (dep[i] > z.D) return fail(ctx, EAGLE_EINVAL, "node deeper than the draft depth");
      if (dep[i] == 1) gen[i] = rank[i];
    }
    std::vector<int> exp((size_t)std::max(1, (z.D - 1) * z.k), 0);
    for (int d = 1; d < z.D; ++d) {
      std::vector<int> rows, expanded;
      for (int i = 0; i < n; ++i) {
        if (dep[i] != d) continue;
        bool has_child = false;
        for (int j = i + 1; j < n && !has_child; ++j) has_child = parent[j] == i;
        if (has_child) expanded.push_back(i);
      }
      if ((int)expanded.size() > z.k) return fail(ctx, EAGLE_EINVAL, "more than k nodes with children at one depth");
      for (int i : expanded) rows.push_back(gen[i]);
      const int lo = d == 1 ? 0 : z.k + (d - 2) * z.k * z.k;
      const int cnt = d == 1 ? z.k : z.k * z.k;
      for (int g = lo; g < lo + cnt && (int)rows.size() < z.k; ++g)
        if (std::find(rows.begin(), rows.end(), g) == rows.end()) rows.push_back(g);
      for (int r = 0; r < z.k; ++r) exp[(size_t)(d - 1) * z.k + r] = rows[r];
      const int base = z.k + (d - 1) * z.k * z.k;
      for (size_t r = 0; r < expanded.size(); ++r)
        for (int j = 0; j < n; ++j)
          if (parent[j] == expanded[r]) gen[j] = base + (int)r * z.k + rank[j];
    }
    std::vector<int> keep(z.NG, 0);
    for (int i = 0; i < n; ++i) {
      if (gen[i] < 0 || gen[i] >= z.NG || keep[gen[i]]) return fail(ctx, EAGLE_EINVAL, "two nodes share a parent and a rank");
      keep[gen[i]] = 1;
    }
    ctx->h_static_exp = exp;
    ctx->h_static_keep = keep;
    if (cudaMemcpyAsync(ctx->static_exp, ctx->h_static_exp.data(), exp.size() * sizeof(int), cudaMemcpyHostToDevice,
                        ctx->st) != cudaSuccess ||
        cudaMemcpyAsync(ctx->static_keep, ctx->h_static_keep.data(), keep.size() * sizeof(int),
                        cudaMemcpyHostToDevice, ctx->st) != cudaSuccess ||
        cudaStreamSynchronize(ctx->st) != cudaSuccess)
      return fail(ctx, EAGLE_ECUDA, "static tree upload failed");
    ctx->static_on = 1;
  }
  ctx->cd.policy = ctx->static_on;
  ctx->cd.static_exp = ctx->static_exp;
  ctx->cd.static_keep = ctx->static_keep;
  if (ctx->graph) { cudaGraphExecDestroy(ctx->graph); ctx->graph = nullptr; }   // the policy is a kernel argument
  return EAGLE_OK;
}

// EAGLE-3 training-time-test forward over one sequence (device int32 x[n]): the target's
// causal pass, then `steps` drafter steps (step 1 causal over sources 0..n-3, later steps
// self-fed with the TTT mask), each scored by its mean token cross-entropy into d_loss[step].
// Uses sequence 0's caches: run eagle_prefill again before cycling.
int eagle_ttt_forward(eagle_ctx* ctx, const int32_t* d_tokens, int n, int steps, float* d_loss) {
  if (!ctx) return EAGLE_EINVAL;
  const Dims& z = ctx->z;
  if (!d_tokens || !d_loss || steps < 1 || steps > 16 || n < steps + 3)
    return fail(ctx, EAGLE_EINVAL, "bad training-time-test arguments");
  if (n > z.P || n - 2 > z.Rd || (size_t)n * steps > (size_t)z.dcap || n > z.cap)
    return fail(ctx, EAGLE_ECAPACITY, "sequence too long for the training-time test in this context");
  if (ctx->graph) { cudaGraphExecDestroy(ctx->graph); ctx->graph = nullptr; }
  ctx->host_ctx_bound = z.max_ctx;   // the cycle state is gone until the next prefill
  ctx->ttt_rows = 0;
  const size_t rb = (size_t)z.H * z.esz;
  // target pass (causal), features of every position
  CK(kv_reserve(ctx, 0, 1, nullptr, 0, n));
  launch_k(ttt_rows_k, (n + 127) / 128, 128, 0, ctx->st, d_tokens, n, 0, n, ctx->row_tok, ctx->row_pos,
           ctx->row_slot, ctx->row_seq, ctx->ttt_tgt, ctx->ctx_len);
  int r = target_forward(ctx, n, ctx->row_tok, ctx->row_pos, ctx->row_slot, ctx->row_seq, n, 0, 0, nullptr, 0,
                         ctx->feat_t, ctx->pre_feat, (size_t)z.max_ctx, 0);
  if (r) return r;
  for (int s = 1; s <= steps; ++s) {
    const int R = s == 1 ? n - 2 : n - 1 - s;
    launch_k(ttt_rows_k, (R + 127) / 128, 128, 0, ctx->st, d_tokens, n, s, R, ctx->row_tok, ctx->row_pos,
             ctx->row_slot, ctx->row_seq, ctx->ttt_tgt, ctx->ctx_len);
    if (s == 1) {
      if (z.kind == 1) {
        r = drafter_forward(ctx, R, ctx->row_tok, ctx->row_pos, ctx->row_slot, ctx->row_seq, R, 2, 0, nullptr, 0,
                            ctx->feat_t, ctx->iota);
      } else {
        r = fuse_rows(ctx, ctx->pre_feat, (size_t)z.max_ctx, nullptr, R);
        if (r) return r;
        r = drafter_forward(ctx, R, ctx->row_tok, ctx->row_pos, ctx->row_slot, ctx->row_seq, R, 2, 0, nullptr, 0,
                            ctx->gbuf, nullptr);
      }
    } else {
      // the previous step's output a (rows 0..R-1 of dout) in place of g; the drafter reads
      // its feature rows before it writes dout
      r = drafter_forward(ctx, R, ctx->row_tok, ctx->row_pos, ctx->row_slot, ctx->row_seq, R, 2, 0, nullptr, 0,
                          ctx->dout, z.kind == 1 ? ctx->iota : nullptr);
    }
    if (r) return r;
    // token loss through the shared LM head, in chunks of the head's row capacity
    for (int r0 = 0; r0 < R; r0 += z.Rh) {
      const int rows = std::min(z.Rh, R - r0);
      HeadParams p = head_params(ctx, rows, 1);
      p.specials = ctx->ttt_tgt + r0;
      p.S = 1;
      p.lse_excl = 0;
      r = lm_head(ctx, (const uint8_t*)ctx->dout + (size_t)r0 * rb, rows, p);
      if (r) return r;
      launch_k(ttt_loss_acc_k, 1, 256, 0, ctx->st, (const float*)ctx->h_lse, (const float*)ctx->h_spec, rows,
               ctx->ttt_acc, r0 == 0 ? 1 : 0, ctx->ttt_ce + r0);
    }
    ctx->ttt_rows = R;
    launch_k(ttt_loss_fin_k, 1, 32, 0, ctx->st, (const float*)ctx->ttt_acc, R, d_loss + (s - 1));
    if (cudaGetLastError() != cudaSuccess) return fail(ctx, EAGLE_ECUDA, "training-time-test launch failed");
  }
  return EAGLE_OK;
}

int eagle_kv_table(const eagle_ctx* ctx, const int32_t** table, int* tab_w, int* n_blocks, int* block) {
  if (!ctx) return EAGLE_EINVAL;
  if (!ctx->page.table) return EAGLE_EUNSUPPORTED;
  if (table) *table = ctx->kv_table;
  if (tab_w) *tab_w = ctx->z.tab_w;
  if (n_blocks) *n_blocks = ctx->z.nblk;
  if (block) *block = 1 << ctx->z.kvb_log2;
  return EAGLE_OK;
}

const char* eagle_last_error(const eagle_ctx* ctx) { return ctx ? ctx->err.c_str() : "null context"; }

void eagle_destroy(eagle_ctx* ctx) {
  if (!ctx) return;
  if (ctx->graph) cudaGraphExecDestroy(ctx->graph);
  for (auto e : ctx->prof_ev) cudaEventDestroy(e);
  for (auto e : ctx->ph_ev) cudaEventDestroy(e);
  delete ctx;
}

}  // extern "C"

namespace eagle {
bool pdl_enabled() {
  static int v = -1;
  if (v < 0) {
    const char* e = getenv("EAGLE_PDL");
    v = (e && e[0] == '0') ? 0 : 1;
  }
  return v == 1;
}
}  // namespace eagle
