// EAGLE-2 dynamic tree on the device: path values, per-depth top-k expansion, global
// top-m rerank, flattening, ancestry bitmask, positions and parent indices.
//
// Path value V_i = product of draft confidences along the root-to-node path, kept as an
// fp32 log-space sum ("EAGLE-2: Context-Aware Dynamic Draft Trees", section "Path Value
// Ranks Prefixes, Not Isolated Tokens", and table "Where It Breaks" on log-space
// ranking). Each depth expands the k best current nodes by (log V desc, generation
// asc); the rerank keeps the m best of all generated nodes by (log V desc, depth asc,
// generation asc), which is ancestor-closed because a confidence never exceeds 1
// (same page, "Global Reranking Separates Exploration from Verification"). Each
// flattened row may see the root, itself and its ancestors only (same page, "The Mask
// Preserves Tree Semantics in One Target Pass").
//
// One CTA per sequence; the selections are warp-level argmax rounds (k of k^2) and a
// rank count over at most a few hundred 64-bit (log V, generation) keys.
#include "common.cuh"
#include "cycle.h"
#include "kernels.h"

namespace eagle {

// Candidates of one drafter row from its LM-head record. Without a special id the head
// ranked the whole vocabulary. With one, the head left it out of the ranking and of the
// lse and reported its logit: if planted it becomes the top-1 with confidence `conf` and
// the others keep their relative mass scaled by 1 - conf; if not planted it is merged
// back into the top-k and into the lse.
__device__ void compose_candidates(const HeadOut& h, int row, int special, bool planted, float conf, int k,
                                   int* out_tok, float* out_logc) {
  const int* ids = h.top_id + (size_t)row * h.K;
  const float* vals = h.top_val + (size_t)row * h.K;
  const float lse = h.lse[row];
  if (special < 0) {
    for (int i = 0; i < k; ++i) { out_tok[i] = ids[i]; out_logc[i] = vals[i] - lse; }
    return;
  }
  if (planted) {
    out_tok[0] = special;
    out_logc[0] = logf(conf);
    const float off = log1pf(-conf);
    for (int i = 1; i < k; ++i) { out_tok[i] = ids[i - 1]; out_logc[i] = vals[i - 1] - lse + off; }
    return;
  }
  const float ls = h.spec_logit[(size_t)row * h.S];
  const float mx = fmaxf(lse, ls);
  const float lse_all = mx + log1pf(expf(-fabsf(lse - ls)));
  int j = 0;
  bool used = false;
  for (int i = 0; i < k; ++i) {
    if (!used && (j >= h.K || rank_before(ls, special, vals[j], ids[j]))) {
      out_tok[i] = special; out_logc[i] = ls - lse_all; used = true;
    } else {
      out_tok[i] = ids[j]; out_logc[i] = vals[j] - lse_all; ++j;
    }
  }
}

__global__ void tree_start_k(CycleDev c) {
  PDL_ENTRY();
  const int b = blockIdx.x;
  const int base = b * c.NG;
  for (int i = threadIdx.x; i < c.NG; i += blockDim.x) c.node_rank[base + i] = -1;
  for (int i = threadIdx.x; i < c.k; i += blockDim.x) {
    c.node_tok[base + i] = c.cand_tok[b * c.kc + i];
    c.node_parent[base + i] = -1;
    c.node_depth[base + i] = 1;
    c.node_logv[base + i] = c.cand_logc[b * c.kc + i];
  }
  if (threadIdx.x == 0) c.n_old[b] = c.ctx_len[b];
}

int tree_start(cudaStream_t st, const CycleDev& c) {
  launch_k(tree_start_k, c.B, 128, 0, st, c);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

// Expansion at depth d: pick the k best depth-d nodes and lay out their drafter rows.
constexpr int TS_QMAX = 8;   // candidates per lane (k * k <= 256)

__global__ void tree_select_k(CycleDev c, int d) {
  PDL_ENTRY();
  const int b = blockIdx.x, lane = threadIdx.x;
  const int base = b * c.NG;
  const int k = c.k;
  const int lo = (d == 1) ? 0 : k + (d - 2) * k * k;
  const int cnt = (d == 1) ? k : k * k;
  if (c.policy == 1) {
    // static tree: the rows expanded at this depth are fixed
    if (lane < k) {
      const int g = c.static_exp[(d - 1) * k + lane];
      c.exp_node[(b * c.D + (d - 1)) * k + lane] = g;
      c.node_rank[base + g] = lane;
    }
  } else {
  // the candidates' path values, loaded once (k <= 16: at most 256 candidates)
  float cv[TS_QMAX];
#pragma unroll
  for (int q = 0; q < TS_QMAX; ++q) cv[q] = lane + 32 * q < cnt ? c.node_logv[base + lo + lane + 32 * q] : -INFINITY;
  uint32_t taken = 0;   // bit q: candidate lo + lane + 32 q already selected
  for (int r = 0; r < k; ++r) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int q = 0; q < TS_QMAX; ++q) {
      if (lane + 32 * q >= cnt || ((taken >> q) & 1)) continue;
      const int g = lo + lane + 32 * q;
      if (rank_before(cv[q], g, bv, bi)) { bv = cv[q]; bi = g; }
    }
    warp_best(bv, bi, bv, bi);
    if (bi != 0x7fffffff && ((bi - lo) & 31) == lane) taken |= 1u << ((bi - lo) >> 5);
    if (lane == 0) {
      c.exp_node[(b * c.D + (d - 1)) * k + r] = bi;
      c.node_rank[base + bi] = r;
    }
  }
  }
  __syncwarp();
  __threadfence_block();
  const int ctx = c.ctx_len[b];
  if (lane < k) {
    const int r = lane;
    const int v = c.exp_node[(b * c.D + (d - 1)) * k + r];
    const int row = b * k + r;
    c.drow_tok[row] = c.node_tok[base + v];
    c.drow_pos[row] = ctx + d - 1;
    c.drow_slot[row] = ctx + (d - 1) * k + r;
    c.drow_seq[row] = b;
    const int par = c.node_parent[base + v];
    c.drow_feat[row] = b * c.fsrc_rows + (d == 1 ? 0 : 1 + (d - 2) * k + c.node_rank[base + par]);
    uint64_t* mw = c.dmask + (size_t)row * c.dmask_words;
    for (int w = 0; w < c.dmask_words; ++w) mw[w] = 0ull;
    int a = v;
    while (a >= 0) {
      const int bit = (c.node_depth[base + a] - 1) * k + c.node_rank[base + a];
      mw[bit >> 6] |= 1ull << (bit & 63);
      a = c.node_parent[base + a];
    }
    int plant = -1;
    if (c.ref && c.on_track[b]) {
      const int cc = c.committed[b];
      if (cc + d < c.ref_len) {
        bool on = true;
        for (int x = v; x >= 0; x = c.node_parent[base + x])
          on = on && (c.ref[(size_t)b * c.ref_len + cc + c.node_depth[base + x] - 1] == c.node_tok[base + x]);
        if (on) plant = c.ref[(size_t)b * c.ref_len + cc + d];
      }
    }
    c.drow_plant[row] = plant;
  }
}

int tree_select(cudaStream_t st, const CycleDev& c, int d) {
  if (c.k > 16) return -1;
  launch_k(tree_select_k, c.B, 32, 0, st, c, d);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

// Children of the depth-d expansion rows: log V_child = log V_parent + log c_child.
__global__ void tree_add_k(CycleDev c, int d, HeadOut h) {
  PDL_ENTRY();
  const int b = blockIdx.x, r = threadIdx.x;
  const int k = c.k;
  if (r >= k) return;
  const int base = b * c.NG;
  const int v = c.exp_node[(b * c.D + (d - 1)) * k + r];
  const int row = b * k + r;
  const int special = c.drow_plant[row];
  const bool planted = special >= 0 &&
                       draw_uniform(c.seed, STREAM_PLANT, (uint32_t)b, c.cycle[b], (uint32_t)(d + 1), 0u) < c.planted_p;
  int tok[16];
  float lc[16];
  compose_candidates(h, row, special, planted, c.planted_conf, k, tok, lc);
  const int g0 = k + (d - 1) * k * k + r * k;
  const float lv = c.node_logv[base + v];
  for (int i = 0; i < k; ++i) {
    c.node_tok[base + g0 + i] = tok[i];
    c.node_parent[base + g0 + i] = v;
    c.node_depth[base + g0 + i] = d + 1;
    c.node_logv[base + g0 + i] = lv + lc[i];
  }
}

int tree_add(cudaStream_t st, const CycleDev& c, int d, const HeadOut& h) {
  if (c.k > 16) return -1;
  launch_k(tree_add_k, c.B, 32, 0, st, c, d, h);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

// Global top-m rerank and flattening.
constexpr int TF_THREADS = 256;

__global__ void __launch_bounds__(TF_THREADS) tree_finalize_k(CycleDev c) {
  PDL_ENTRY();
  extern __shared__ uint8_t sm[];
  const int NG = c.NG;
  uint64_t* key = reinterpret_cast<uint64_t*>(sm);
  int* row_of = reinterpret_cast<int*>(key + NG);
  const int b = blockIdx.x;
  const int base = b * c.NG;
  for (int i = threadIdx.x; i < NG; i += blockDim.x)
    key[i] = ((uint64_t)(~f32_order_key(c.node_logv[base + i])) << 32) | (uint32_t)i;
  __syncthreads();
  for (int i = threadIdx.x; i < NG; i += blockDim.x) {
    if (c.policy == 1) {   // static tree: the kept nodes are fixed
      row_of[i] = c.static_keep[i] ? 1 : 0;
      continue;
    }
    const uint64_t ki = key[i];
    int rank = 0;
    for (int j = 0; j < NG; ++j) rank += key[j] < ki;
    row_of[i] = rank < c.m ? 1 : 0;
  }
  __syncthreads();
  // flattened row = 1 + number of kept nodes with a smaller generation index: each thread
  // counts a contiguous run of nodes, an exclusive block scan gives its runs' offsets
  {
    __shared__ int s_warp[TF_THREADS / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int per = (NG + TF_THREADS - 1) / TF_THREADS;
    const int i0 = min(NG, threadIdx.x * per), i1 = min(NG, i0 + per);
    int cnt = 0;
    for (int i = i0; i < i1; ++i) cnt += row_of[i];
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    int run = incl - cnt;
    for (int w = 0; w < warp; ++w) run += s_warp[w];
    for (int i = i0; i < i1; ++i) {
      const int kept = row_of[i];
      key[i] = (uint64_t)(kept ? 1 + run : 0);
      run += kept;
    }
  }
  __syncthreads();
  const int T1 = c.T1;
  // the tree rows' parent and token, kept in shared memory for the mask and child walks
  int* s_par = row_of + NG;
  int* s_tok = s_par + T1;
  for (int i = threadIdx.x; i < NG; i += blockDim.x) row_of[i] = key[i] ? (int)key[i] : -1;
  for (int r = threadIdx.x; r < T1; r += blockDim.x) { s_par[r] = -1; s_tok[r] = -1; }
  __syncthreads();
  const int ctx = c.ctx_len[b];
  const int rb = b * T1;
  if (threadIdx.x == 0) {
    s_tok[0] = c.root_tok[b];
    c.tree_tok[rb] = c.root_tok[b];
    c.tree_pos[rb] = ctx;
    c.tree_slot[rb] = ctx;
    c.tree_seq[rb] = b;
    c.tree_parent[rb] = -1;
    c.tree_node[rb] = -1;
  }
  for (int i = threadIdx.x; i < NG; i += blockDim.x) {
    const int r = row_of[i];
    if (r < 0) continue;
    if (r >= T1) { latch_error(c.err, DEVERR_BOUNDS); continue; }
    const int p = c.node_parent[base + i];
    int pr = 0;
    if (p >= 0) {
      pr = row_of[p];
      if (pr < 0) { latch_error(c.err, DEVERR_BOUNDS); pr = 0; }
    }
    const int tok = c.node_tok[base + i];
    s_par[r] = pr;
    s_tok[r] = tok;
    c.tree_tok[rb + r] = tok;
    c.tree_pos[rb + r] = ctx + c.node_depth[base + i];
    c.tree_slot[rb + r] = ctx + r;
    c.tree_seq[rb + r] = b;
    c.tree_parent[rb + r] = pr;
    c.tree_node[rb + r] = i;
  }
  __syncthreads();
  // ancestry masks built in registers (T1 <= 256: at most four words), written once
  for (int r = threadIdx.x; r < T1; r += blockDim.x) {
    uint64_t m0 = 0ull, m1 = 0ull, m2 = 0ull, m3 = 0ull;
    int a = r, guard = 0;
    while (a >= 0 && guard++ <= T1) {
      const uint64_t bit = 1ull << (a & 63);
      const int w = a >> 6;
      m0 |= w == 0 ? bit : 0ull;
      m1 |= w == 1 ? bit : 0ull;
      m2 |= w == 2 ? bit : 0ull;
      m3 |= w == 3 ? bit : 0ull;
      a = s_par[a];
    }
    uint64_t* mw = c.tmask + (size_t)(rb + r) * c.tmask_words;
    mw[0] = m0;
    if (c.tmask_words > 1) mw[1] = m1;
    if (c.tmask_words > 2) mw[2] = m2;
    if (c.tmask_words > 3) mw[3] = m3;
    int n = 0;
    int* kids = c.tree_kids + (size_t)(rb + r) * c.k;
    for (int x = r + 1; x < T1 && n < c.k; ++x)
      if (s_par[x] == r) kids[n++] = s_tok[x];
    for (; n < c.k; ++n) kids[n] = -1;
  }
}

int tree_finalize(cudaStream_t st, const CycleDev& c) {
  if (c.m > c.NG || c.T1 > 256 || c.tmask_words > 4) return -1;
  const size_t sm = (size_t)c.NG * (sizeof(uint64_t) + sizeof(int)) + (size_t)2 * c.T1 * sizeof(int);
  launch_k(tree_finalize_k, c.B, TF_THREADS, sm, st, c);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

// Row whose drafter output feeds the root's next candidates, and its planted token.
__global__ void root_prepare_k(CycleDev c, int rows_per_seq, int* root_row) {
  PDL_ENTRY();
  const int b = blockIdx.x;
  if (threadIdx.x) return;
  root_row[b] = b * rows_per_seq + c.acc_len[b];
  int plant = -1;
  if (c.ref && c.on_track[b]) {
    const int cc = c.committed[b];
    if (cc < c.ref_len) plant = c.ref[(size_t)b * c.ref_len + cc];
  }
  c.root_plant[b] = plant;
}

int root_prepare(cudaStream_t st, const CycleDev& c, int rows_per_seq, int* root_row) {
  launch_k(root_prepare_k, c.B, 32, 0, st, c, rows_per_seq, root_row);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

// Depth-1 candidates of the root for the next cycle (`advance` = 1 after a cycle, 0 at
// prefill); the planted draw is keyed by the cycle that will use them.
__global__ void root_candidates_k(CycleDev c, HeadOut h, int seq_lo, int advance) {
  PDL_ENTRY();
  const int b = seq_lo + blockIdx.x;
  const int row = blockIdx.x;
  if (threadIdx.x == 0) {
    const uint32_t cyc = c.cycle[b] + (uint32_t)advance;
    const int special = c.root_plant[b];
    const bool planted =
        special >= 0 && draw_uniform(c.seed, STREAM_PLANT, (uint32_t)b, cyc, 1u, 0u) < c.planted_p;
    int tok[16];
    float lc[16];
    compose_candidates(h, row, special, planted, c.planted_conf, c.kc, tok, lc);
    for (int i = 0; i < c.kc; ++i) {
      c.cand_tok[b * c.kc + i] = tok[i];
      c.cand_logc[b * c.kc + i] = lc[i];
    }
    c.cycle[b] = cyc;
  }
}

int root_candidates(cudaStream_t st, const CycleDev& c, const HeadOut& h, int advance) {
  launch_k(root_candidates_k, c.B, 32, 0, st, c, h, 0, advance);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

int root_candidates_seq(cudaStream_t st, const CycleDev& c, const HeadOut& h, int seq) {
  launch_k(root_candidates_k, 1, 32, 0, st, c, h, seq, 0);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace eagle
