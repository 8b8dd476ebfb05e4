// Device-side state of the cycle shared by the tree, acceptance and row-setup kernels.
// All arrays live in the caller's workspace; this struct only carries pointers and sizes.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "kernels.h"

namespace eagle {

struct CycleDev {
  int B, k, D, m, T1, NG, V;
  int kc;                   // root candidates kept per sequence (>= k; the tree uses the first k)
  int dmask_words, tmask_words;
  int fsrc_rows;            // 1 + (D - 1) * k feature rows per sequence (row 0 = root feature)
  // tree policy: 0 = EAGLE-2 dynamic (expand by path value, rerank the top m); 1 = static
  // (EAGLE-1): the expansion rows and the kept nodes are fixed in advance
  int policy;
  const int* static_exp;    // [D - 1][k] generation index expanded by row r at depth d
  const int* static_keep;   // [NG] 1 = node kept (exactly m of them)
  // per-sequence state
  int* ctx_len;             // [B] target (and drafter) KV length n
  int* n_old;               // [B] n at the start of the running cycle
  int* root_tok;            // [B] last committed token (not yet in the KV cache)
  int* committed;           // [B] tokens committed since prefill (the prefill token included)
  const int* stop_at;       // [B] a sequence with committed >= stop_at is finished (INT32_MAX: none)
  int* on_track;            // [B] committed tokens equal the planted reference so far
  uint32_t* cycle;          // [B] cycle counter (Philox field)
  const int* ref;           // [B][ref_len] planted reference continuation (null: not planted)
  int ref_len;
  float planted_p, planted_conf, inv_t;
  uint64_t seed;
  int sampling;             // 1 = speculative sampling, 0 = greedy
  // depth-1 candidates of the root, in rank order
  int* cand_tok;            // [B][kc]
  float* cand_logc;         // [B][kc]
  int* root_plant;          // [B] planted-candidate id for the root's drafter row (-1 none)
  // node table (generation order)
  int* node_tok;            // [B][NG]
  int* node_parent;         // [B][NG] (-1 = child of the root)
  int* node_depth;          // [B][NG]
  float* node_logv;         // [B][NG]
  int* node_rank;           // [B][NG] expansion rank within its depth, -1 if never expanded
  int* exp_node;            // [B][D][k]
  // drafter expansion rows (B * k)
  int* drow_tok;
  int* drow_pos;
  int* drow_slot;
  int* drow_seq;
  int* drow_feat;           // feature-source row (into the [B][fsrc_rows][H] buffer)
  int* drow_plant;          // planted-candidate id for the row's children (-1 none)
  uint64_t* dmask;          // [B*k][dmask_words]
  // flattened tree (B * T1 rows)
  int* tree_tok;
  int* tree_pos;
  int* tree_slot;
  int* tree_seq;
  int* tree_parent;
  int* tree_node;
  int* tree_kids;           // [B*T1][k] children tokens in rank order (-1 padded)
  uint64_t* tmask;          // [B*T1][tmask_words]
  // acceptance
  int* acc_len;             // [B]
  int* emitted;             // [B] tokens committed by the cycle (0 for a finished sequence)
  int* acc_path;            // [B][D] accepted flattened rows
  int* bonus;               // [B]
  float* margin;            // [B][T1] greedy top-2 margin per verify row (diagnostic)
  int* err;
};

// LM-head outputs for a group of rows (K entries per row).
struct HeadOut {
  const int* top_id;
  const float* top_val;
  const float* lse;
  const float* spec_logit;  // [rows][S]
  int K, S;
};

int tree_start(cudaStream_t st, const CycleDev& c);
int tree_select(cudaStream_t st, const CycleDev& c, int d);
int tree_add(cudaStream_t st, const CycleDev& c, int d, const HeadOut& h);
int tree_finalize(cudaStream_t st, const CycleDev& c);
int accept_walk(cudaStream_t st, const CycleDev& c, const HeadOut& h, int* out_tokens, int* out_count);
// accepted tree slots n + acc_path[j] -> n + 1 + j, every layer (layer_elems apart)
int compact_kv(cudaStream_t st, int dtype, void* kc, void* vc, int layers, size_t layer_elems, int B, int nkv,
               int cap, int d, const int* n_old, const int* acc_len, const int* acc_path, int Dmax,
               const KvPage& page);
// drafter update rows after acceptance: rows b*(D+1)+j, j = 0..D
int update_rows(cudaStream_t st, const CycleDev& c, int* row_tok, int* row_pos, int* row_slot, int* row_seq,
                int* row_featsrc);
int root_prepare(cudaStream_t st, const CycleDev& c, int rows_per_seq, int* root_row);
int root_candidates(cudaStream_t st, const CycleDev& c, const HeadOut& h, int advance);
// plain decoding / prefill helpers
int plain_rows(cudaStream_t st, const CycleDev& c, int* row_tok, int* row_pos, int* row_slot, int* row_seq);
int plain_advance(cudaStream_t st, const CycleDev& c, const int* next_tok, int K, const float* top_val, int* out,
                  float* margin, int ld_out, int step);
int prefill_rows(cudaStream_t st, const int* prompt, int seq, int p0, int n, int last_tok_from_root,
                 const int* root_tok, int* row_tok, int* row_pos, int* row_slot, int* row_seq, int shift);
int prefill_finish(cudaStream_t st, const CycleDev& c, int seq, int n, const int* first_tok);
int prefill_rows_batched(cudaStream_t st, const int* tokens, int B, int n, int shift, const int* root_tok,
                         int* row_tok, int* row_pos, int* row_slot, int* row_seq);
int prefill_finish_batched(cudaStream_t st, const CycleDev& c, int n, const int* first_tok, int K);

}  // namespace eagle
