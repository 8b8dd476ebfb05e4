// Acceptance walk along the verified tree, KV-cache compaction of the accepted path,
// and the row set-up kernels of the drafter update, plain decoding and prefill.
//
// Acceptance keeps drafted tokens from the root while they pass the test (equal to the
// target's argmax when greedy, the rejection-sampling rule when sampling) and takes the
// target's own token at the first rejection ("EAGLE: Feature-Level Drafting", list
// "Speculative decoding in four moves", items 3-4; "EAGLE-2: Context-Aware Dynamic
// Draft Trees", table "Putting It Together", step 5). The multi-candidate sampling rule
// used is recursive point-mass rejection: at node u the kept children are tried in draft
// rank order and child t is accepted when U * (1 - sum of p over tried children) < p(t),
// U a Philox uniform keyed by (seed; try index, row, cycle, sequence); if all are
// rejected the bonus is the Gumbel-argmax of p over the vocabulary minus those children,
// computed inside the LM-head epilogue.
#include "common.cuh"
#include "cycle.h"
#include "kernels.h"

namespace eagle {

__global__ void accept_k(CycleDev c, HeadOut h, int* out_tokens, int* out_count) {
  PDL_ENTRY();
  const int b = blockIdx.x;
  const int T1 = c.T1, rb = b * T1;
  // greedy top-2 margins (diagnostic for near-ties)
  if (!c.sampling && h.K >= 2 && c.margin)
    for (int r = threadIdx.x; r < T1; r += blockDim.x)
      c.margin[rb + r] = h.top_val[(size_t)(rb + r) * h.K] - h.top_val[(size_t)(rb + r) * h.K + 1];
  if (threadIdx.x) return;
  const int cc = c.committed[b];
  const int stop = c.stop_at ? c.stop_at[b] : INT32_MAX;
  if (cc >= stop) {
    // finished: masked out of this and every later cycle, its state left as it is (its rows
    // still go through the fixed-shape cycle; nothing of them is committed)
    c.acc_len[b] = 0;
    c.bonus[b] = c.root_tok[b];
    c.n_old[b] = c.ctx_len[b];
    c.emitted[b] = 0;
    if (out_count) out_count[b] = 0;
    return;
  }
  int u = 0, L = 0, bonus = -1;
  while (true) {
    const int row = rb + u;
    int next = -1;
    if (!c.sampling) {
      const int a = h.top_id[(size_t)row * h.K];
      for (int x = u + 1; x < T1; ++x)
        if (c.tree_parent[rb + x] == u && c.tree_tok[rb + x] == a) { next = x; break; }
      if (next < 0 || L >= c.D) { bonus = a; break; }
    } else {
      float tried = 0.f;
      int i = 0;
      for (int x = u + 1; x < T1 && i < c.k; ++x) {
        if (c.tree_parent[rb + x] != u) continue;
        const float pt = expf(h.spec_logit[(size_t)row * h.S + i] * c.inv_t - h.lse[row]);
        const float U = draw_uniform(c.seed, STREAM_ACCEPT, (uint32_t)b, c.cycle[b], (uint32_t)i, (uint32_t)u);
        if (U * (1.f - tried) < pt) { next = x; break; }
        tried += pt;
        ++i;
      }
      if (next < 0 || L >= c.D) { bonus = h.top_id[(size_t)row * h.K]; break; }
    }
    c.acc_path[b * c.D + L] = next;
    ++L;
    u = next;
  }
  c.acc_len[b] = L;
  c.bonus[b] = bonus;
  int on = c.on_track[b];
  for (int j = 0; j <= L; ++j) {
    const int t = j < L ? c.tree_tok[rb + c.acc_path[b * c.D + j]] : bonus;
    if (out_tokens) out_tokens[b * (c.D + 1) + j] = t;
    if (c.ref) on = on && (cc + j < c.ref_len) && c.ref[(size_t)b * c.ref_len + cc + j] == t;
  }
  // the last cycle of a sequence with a limit emits only up to the limit
  const int emit = min(L + 1, stop - cc);
  c.emitted[b] = emit;
  if (out_count) out_count[b] = emit;
  c.on_track[b] = on;
  c.committed[b] = cc + L + 1;
  c.root_tok[b] = bonus;
  c.ctx_len[b] = c.n_old[b] + L + 1;
}

int accept_walk(cudaStream_t st, const CycleDev& c, const HeadOut& h, int* out_tokens, int* out_count) {
  launch_k(accept_k, c.B, 64, 0, st, c, h, out_tokens, out_count);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

// slot n + j <- slot n + path[j - 1], j = 1..L, in every layer. Each thread owns fixed
// element positions and reads all L sources before writing any target, so overlapping
// source/target slots cannot race.
template <typename T>
__global__ void compact_k(T* kc, T* vc, int layers, size_t layer_elems, int B, int nkv, int cap, int d,
                          const int* n_old, const int* acc_len, const int* acc_path, int Dmax, KvPage page) {
  PDL_ENTRY();
  const int layer = blockIdx.x;
  const int bh = blockIdx.y;
  const int b = bh / nkv, h = bh - b * nkv;
  const int L = acc_len[b];
  if (L <= 0) return;
  const int n = n_old[b];
  T* kl = kc + (size_t)layer * layer_elems;
  T* vl = vc + (size_t)layer * layer_elems;
  T tk[8], tv[8];
  for (int e = threadIdx.x; e < d; e += blockDim.x) {
    for (int j = 0; j < L && j < 8; ++j) {
      const size_t s = kv_row(page, b, nkv, h, cap, n + acc_path[b * Dmax + j]) * d + e;
      tk[j] = kl[s];
      tv[j] = vl[s];
    }
    for (int j = 0; j < L && j < 8; ++j) {
      const size_t t = kv_row(page, b, nkv, h, cap, n + 1 + j) * d + e;
      kl[t] = tk[j];
      vl[t] = tv[j];
    }
  }
}

int compact_kv(cudaStream_t st, int dtype, void* kc, void* vc, int layers, size_t layer_elems, int B, int nkv,
               int cap, int d, const int* n_old, const int* acc_len, const int* acc_path, int Dmax,
               const KvPage& page) {
  if (Dmax > 8) return -1;
  dim3 grid(layers, B * nkv);
  if (dtype == DT_F32)
    launch_k(compact_k<float>, grid, 128, 0, st, (float*)kc, (float*)vc, layers, layer_elems, B, nkv, cap, d, n_old,
             acc_len, acc_path, Dmax, page);
  else
    launch_k(compact_k<__nv_bfloat16>, grid, 128, 0, st, (__nv_bfloat16*)kc, (__nv_bfloat16*)vc, layers, layer_elems, B,
             nkv, cap, d, n_old, acc_len, acc_path, Dmax, page);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

// Drafter rows after acceptance: drafter position n + j carries (feature of target
// position n + j, token at n + j + 1), j = 0..L; rows L+1..D are padding whose outputs
// are ignored and whose KV lands beyond the new context.
__global__ void update_rows_k(CycleDev c, int* row_tok, int* row_pos, int* row_slot, int* row_seq,
                              int* row_featsrc) {
  PDL_ENTRY();
  const int b = blockIdx.x, j = threadIdx.x;
  if (j > c.D) return;
  const int L = c.acc_len[b];
  const int jj = j < L ? j : L;
  const int tr = jj == 0 ? 0 : c.acc_path[b * c.D + jj - 1];
  const int row = b * (c.D + 1) + j;
  row_featsrc[row] = b * c.T1 + tr;
  row_tok[row] = jj < L ? c.tree_tok[b * c.T1 + c.acc_path[b * c.D + jj]] : c.bonus[b];
  row_pos[row] = c.n_old[b] + j;
  row_slot[row] = c.n_old[b] + j;
  row_seq[row] = b;
}

int update_rows(cudaStream_t st, const CycleDev& c, int* row_tok, int* row_pos, int* row_slot, int* row_seq,
                int* row_featsrc) {
  if (c.D + 1 > 32) return -1;
  launch_k(update_rows_k, c.B, 32, 0, st, c, row_tok, row_pos, row_slot, row_seq, row_featsrc);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

__global__ void plain_rows_k(CycleDev c, int* row_tok, int* row_pos, int* row_slot, int* row_seq) {
  PDL_ENTRY();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= c.B) return;
  row_tok[b] = c.root_tok[b];
  row_pos[b] = c.ctx_len[b];
  row_slot[b] = c.ctx_len[b];
  row_seq[b] = b;
}

int plain_rows(cudaStream_t st, const CycleDev& c, int* row_tok, int* row_pos, int* row_slot, int* row_seq) {
  launch_k(plain_rows_k, (c.B + 127) / 128, 128, 0, st, c, row_tok, row_pos, row_slot, row_seq);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

__global__ void plain_advance_k(CycleDev c, const int* next_tok, int K, const float* top_val, int* out,
                                float* margin, int ld_out, int step) {
  PDL_ENTRY();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= c.B) return;
  const int t = next_tok[b * K];
  if (out) out[(size_t)b * ld_out + step] = t;
  if (margin) margin[(size_t)b * ld_out + step] = K >= 2 ? top_val[b * K] - top_val[b * K + 1] : NAN;
  c.root_tok[b] = t;
  c.ctx_len[b] += 1;
}

int plain_advance(cudaStream_t st, const CycleDev& c, const int* next_tok, int K, const float* top_val, int* out,
                  float* margin, int ld_out, int step) {
  launch_k(plain_advance_k, (c.B + 127) / 128, 128, 0, st, c, next_tok, K, top_val, out, margin, ld_out, step);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

// Prefill rows p0 .. p0+n-1 of one sequence. shift = 0: target rows (token p); shift = 1:
// drafter rows (token p + 1, the first generated token for the last prompt position).
__global__ void prefill_rows_k(const int* prompt, int n_total, int seq, int p0, int n, int shift,
                               const int* root_tok, int* row_tok, int* row_pos, int* row_slot, int* row_seq) {
  PDL_ENTRY();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int p = p0 + i;
  row_tok[i] = shift ? (p + 1 < n_total ? prompt[p + 1] : root_tok[seq]) : prompt[p];
  row_pos[i] = p;
  row_slot[i] = p;
  row_seq[i] = seq;
}

int prefill_rows(cudaStream_t st, const int* prompt, int seq, int p0, int n, int n_total_shift,
                 const int* root_tok, int* row_tok, int* row_pos, int* row_slot, int* row_seq, int shift) {
  if (n <= 0) return 0;
  launch_k(prefill_rows_k, (n + 127) / 128, 128, 0, st, prompt, n_total_shift, seq, p0, n, shift, root_tok, row_tok,
                                                  row_pos, row_slot, row_seq);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

__global__ void prefill_finish_k(CycleDev c, int seq, int n, const int* first_tok) {
  PDL_ENTRY();
  if (threadIdx.x) return;
  const int t = first_tok[0];
  c.root_tok[seq] = t;
  c.committed[seq] = 1;
  const int on = c.ref ? (c.ref_len > 0 && c.ref[(size_t)seq * c.ref_len] == t) : 1;
  c.on_track[seq] = on;
  c.ctx_len[seq] = n;
  c.n_old[seq] = n;
  c.acc_len[seq] = 0;
  c.cycle[seq] = 0;
  c.root_plant[seq] = (c.ref && on && 1 < c.ref_len) ? c.ref[(size_t)seq * c.ref_len + 1] : -1;
}

// Batched prefill rows for B equal-length prompts (row b * n + p): shift as above.
__global__ void prefill_rows_batched_k(const int* tokens, int B, int n, int shift, const int* root_tok, int* row_tok,
                                       int* row_pos, int* row_slot, int* row_seq) {
  PDL_ENTRY();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= B * n) return;
  const int b = i / n, p = i % n;
  row_tok[i] = shift ? (p + 1 < n ? tokens[b * n + p + 1] : root_tok[b]) : tokens[b * n + p];
  row_pos[i] = p;
  row_slot[i] = p;
  row_seq[i] = b;
}

int prefill_rows_batched(cudaStream_t st, const int* tokens, int B, int n, int shift, const int* root_tok,
                         int* row_tok, int* row_pos, int* row_slot, int* row_seq) {
  launch_k(prefill_rows_batched_k, (B * n + 127) / 128, 128, 0, st, tokens, B, n, shift, root_tok, row_tok, row_pos,
           row_slot, row_seq);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

__global__ void prefill_finish_batched_k(CycleDev c, int n, const int* first_tok, int K) {
  PDL_ENTRY();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= c.B) return;
  const int t = first_tok[b * K];
  c.root_tok[b] = t;
  c.committed[b] = 1;
  const int on = c.ref ? (c.ref_len > 0 && c.ref[(size_t)b * c.ref_len] == t) : 1;
  c.on_track[b] = on;
  c.ctx_len[b] = n;
  c.n_old[b] = n;
  c.acc_len[b] = 0;
  c.cycle[b] = 0;
  c.root_plant[b] = (c.ref && on && 1 < c.ref_len) ? c.ref[(size_t)b * c.ref_len + 1] : -1;
}

int prefill_finish_batched(cudaStream_t st, const CycleDev& c, int n, const int* first_tok, int K) {
  launch_k(prefill_finish_batched_k, (c.B + 127) / 128, 128, 0, st, c, n, first_tok, K);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

int prefill_finish(cudaStream_t st, const CycleDev& c, int seq, int n, const int* first_tok) {
  launch_k(prefill_finish_k, 1, 32, 0, st, c, seq, n, first_tok);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace eagle
