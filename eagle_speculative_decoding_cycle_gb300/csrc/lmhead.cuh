// Fused LM-head epilogue: per (vocab tile, row) partial softmax statistics and top-K.
//
// The LM head is "a single matrix followed by softmax" ("EAGLE: Feature-Level
// Drafting", section "The big idea: draft at the feature level"). Instead of writing
// full-vocabulary logits, each 128-wide vocabulary tile reduces its logits per row to
// a record (running max, sum of exp relative to that max, and the K best entries by a
// ranking value). A second kernel merges the records of all tiles in a fixed order.
// The same routine serves three uses:
//   drafter top-k + confidence: rank = logit, lse over all but the planted candidate;
//   greedy verify: K = 2 (argmax and top-2 margin);
//   sampling verify: rank = logit/T + Gumbel noise, the row's kept children excluded
//   from the ranking (their logits are reported separately), lse over everything.
#pragma once

#include "common.cuh"

struct HeadParams {
  int vocab;
  int n_rows;            // rows (tokens) of this launch
  int K;                 // entries kept per row, 1..16
  float inv_t;           // logits are scaled by this for lse and ranking
  int gumbel;            // add Gumbel(0,1) noise to the ranking value
  int lse_excl;          // leave the special ids out of max / sum-exp
  const int* specials;   // [n_rows][S] ids excluded from ranking (-1 = unused), or null
  int S;
  float* spec_logit;     // [n_rows][S] raw logit of each special id (written by its tile)
  const int* row_seq;    // Philox sequence field per row (null = seq_base)
  int seq_base;
  const int* row_key;    // Philox row field per row (null = row % key_mod, or row if key_mod = 0)
  int key_mod;
  const uint32_t* cycle; // cycle counter(s) on the device (null = cycle_const)
  int cycle_per_seq;     // 1: cycle[seq], 0: cycle[0]
  uint32_t cycle_const;
  uint32_t stream;       // Philox stream id of the Gumbel draws
  uint64_t seed;
  float* part;           // [n_tiles][n_rows][2 + 2K] partial records
  int n_tiles;
  int* top_id;           // merge outputs: [n_rows][K]
  float* top_val;        // [n_rows][K] ranking values
  float* lse;            // [n_rows]
};

EAGLE_DEV float gumbel_noise(const HeadParams& p, int row, int id) {
  const uint32_t seq = p.row_seq ? (uint32_t)p.row_seq[row] : (uint32_t)p.seq_base;
  const uint32_t key = p.row_key ? (uint32_t)p.row_key[row]
                                 : (p.key_mod ? (uint32_t)(row % p.key_mod) : (uint32_t)row);
  const uint32_t cyc = p.cycle ? (p.cycle_per_seq ? p.cycle[seq] : p.cycle[0]) : p.cycle_const;
  u32x4 o = philox4x32_10(u32x4{(uint32_t)id >> 2, key, cyc, (seq << 8) | p.stream},
                          (uint32_t)p.seed, (uint32_t)(p.seed >> 32));
  const uint32_t w = (id & 3) == 0 ? o.x : (id & 3) == 1 ? o.y : (id & 3) == 2 ? o.z : o.w;
  const float u = philox_uniform(w);
  return -logf(-logf(u));
}

// One warp reduces the 128 logits `vals` (shared memory) of vocabulary tile `tile`
// for row `row` into its partial record.
EAGLE_DEV void head_tile_row(const float* vals, int tile, int row, const HeadParams& p, int lane) {
  float rv[4];
  int rid[4];
  float mx = -INFINITY;
  float sv[4];
  bool in_lse[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int i = lane + 32 * q;
    const int id = tile * 128 + i;
    const bool valid = id < p.vocab;
    const float x = vals[i];
    bool special = false;
    if (valid && p.specials) {
      for (int s = 0; s < p.S; ++s) {
        if (p.specials[row * p.S + s] == id) {
          special = true;
          p.spec_logit[row * p.S + s] = x;
        }
      }
    }
    sv[q] = x * p.inv_t;
    in_lse[q] = valid && !(special && p.lse_excl);
    if (in_lse[q]) mx = fmaxf(mx, sv[q]);
    const bool rank_ok = valid && !special;
    rv[q] = rank_ok ? (p.gumbel ? sv[q] + gumbel_noise(p, row, id) : sv[q]) : -INFINITY;
    rid[q] = rank_ok ? id : 0x7fffffff;
  }
  mx = key2f(__reduce_max_sync(0xffffffffu, f2key(mx)));
  float se = 0.f;
  if (mx != -INFINITY) {
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (in_lse[q]) se += expf(sv[q] - mx);
  }
  se = warp_sum(se);
  float* rec = p.part + ((size_t)tile * p.n_rows + row) * (2 + 2 * p.K);
  if (lane == 0) {
    rec[0] = mx;
    rec[1] = se;
  }
  for (int k = 0; k < p.K; ++k) {
    // lane's best remaining candidate
    float bv = rv[0];
    int bi = rid[0];
#pragma unroll
    for (int q = 1; q < 4; ++q)
      if (rank_before(rv[q], rid[q], bv, bi)) { bv = rv[q]; bi = rid[q]; }
    warp_best(bv, bi, bv, bi);
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (rid[q] == bi) { rv[q] = -INFINITY; rid[q] = 0x7fffffff; }
    if (lane == 0) {
      rec[2 + 2 * k] = bv;
      rec[3 + 2 * k] = __int_as_float(bi == 0x7fffffff ? -1 : bi);
    }
  }
}

// The same record built by one thread from 32 consecutive vocabulary entries of one row
// (ids id0 .. id0 + 31, unit stride in shared memory): the tensor-core epilogue gives each
// lane one token column and each warp one quarter of the 128-entry tile, so the reduction
// needs no cross-lane step. head_quarter_load reads the entries into registers (max and sum
// of exp over the entries in the lse, ranking values); head_quarter_select then takes the K
// kept entries in K rounds, each the best remaining entry in the rank_before order (the
// scan runs in id order and keeps the first of equal values), and writes the quarter's
// record [m, s, (value, id) x K] (id -1: empty) to shared memory. head_quarter_merge
// combines the four quarter records of a row in quarter order into the tile's record.
EAGLE_DEV void head_quarter_load(const float* vals, int id0, int row, const HeadParams& p, float (&r)[32],
                                 uint32_t& rank_ok, float& mx, float& se) {
  uint32_t special = 0;
  if (p.specials) {
    for (int s = 0; s < p.S; ++s) {
      const int sid = p.specials[row * p.S + s];
      const int o = sid - id0;
      if (o >= 0 && o < 32 && sid < p.vocab) {
        special |= 1u << o;
        p.spec_logit[row * p.S + s] = vals[o];
      }
    }
  }
  const uint32_t valid = (p.vocab - id0 >= 32) ? 0xffffffffu : ((1u << max(0, p.vocab - id0)) - 1u);
  const uint32_t in_lse = p.lse_excl ? (valid & ~special) : valid;
  rank_ok = valid & ~special;
  mx = -INFINITY;
#pragma unroll
  for (int v = 0; v < 32; ++v) {
    r[v] = vals[v] * p.inv_t;
    if ((in_lse >> v) & 1u) mx = fmaxf(mx, r[v]);
  }
  se = 0.f;
  if (mx != -INFINITY) {
#pragma unroll
    for (int v = 0; v < 32; ++v)
      if ((in_lse >> v) & 1u) se += expf(r[v] - mx);
  }
  if (p.gumbel) {
#pragma unroll
    for (int v = 0; v < 32; ++v)
      if ((rank_ok >> v) & 1u) r[v] += gumbel_noise(p, row, id0 + v);
  }
}

EAGLE_DEV void head_quarter_select(const float (&r)[32], uint32_t avail, int id0, int K, float mx, float se,
                                   float* dst) {
  dst[0] = mx;
  dst[1] = se;
  for (int k = 0; k < K; ++k) {
    float bv = -INFINITY;
    int bvi = -1;
#pragma unroll
    for (int v = 0; v < 32; ++v)
      if (((avail >> v) & 1u) && (bvi < 0 || r[v] > bv)) { bv = r[v]; bvi = v; }
    if (bvi >= 0) avail &= ~(1u << bvi);
    dst[2 + 2 * k] = bvi >= 0 ? bv : -INFINITY;
    dst[3 + 2 * k] = __int_as_float(bvi >= 0 ? id0 + bvi : -1);
  }
}

// q0 .. q3: the four quarter records of the row, in quarter order.
EAGLE_DEV void head_quarter_merge(const float* q0, const float* q1, const float* q2, const float* q3, int K,
                                  int tile, int row, const HeadParams& p) {
  const float* qs[4] = {q0, q1, q2, q3};
  float M = -INFINITY, S = 0.f;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float m2 = qs[q][0], s2 = qs[q][1];
    if (m2 != -INFINITY) {
      if (m2 > M) { S = S * expf(M - m2) + s2; M = m2; }
      else S += s2 * expf(m2 - M);
    }
  }
  float* rec = p.part + ((size_t)tile * p.n_rows + row) * (2 + 2 * K);
  rec[0] = M;
  rec[1] = S;
  int h0 = 0, h1 = 0, h2 = 0, h3 = 0;     // next entry of each quarter's sorted list
  for (int k = 0; k < K; ++k) {
    float bv = -INFINITY;
    int bi = 0x7fffffff, bq = -1;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int h = q == 0 ? h0 : q == 1 ? h1 : q == 2 ? h2 : h3;
      if (h < K) {
        const float cv = qs[q][2 + 2 * h];
        const int ci = __float_as_int(qs[q][3 + 2 * h]);
        if (ci >= 0 && (bq < 0 || rank_before(cv, ci, bv, bi))) { bv = cv; bi = ci; bq = q; }
      }
    }
    h0 += bq == 0;
    h1 += bq == 1;
    h2 += bq == 2;
    h3 += bq == 3;
    rec[2 + 2 * k] = bq >= 0 ? bv : -INFINITY;
    rec[3 + 2 * k] = __int_as_float(bq >= 0 ? bi : -1);
  }
}

// Merge: each thread folds the records of tiles t0, t0 + stride, ... into its sorted
// list (lv, li; K entries, the rest -inf) and its (max, sum-exp) pair. A thread's first
// record is taken as is (records are sorted); later ones are inserted.
EAGLE_DEV void head_merge_fold(const HeadParams& p, int row, int t0, int stride, float* lv, int* li, float& M,
                               float& S) {
  const int K = p.K;
#pragma unroll
  for (int k = 0; k < 16; ++k) { lv[k] = -INFINITY; li[k] = 0x7fffffff; }
  M = -INFINITY;
  S = 0.f;
  for (int t = t0; t < p.n_tiles; t += stride) {
    const float* rec = p.part + ((size_t)t * p.n_rows + row) * (2 + 2 * K);
    const float m2 = rec[0], s2 = rec[1];
    if (m2 != -INFINITY) {
      if (m2 > M) { S = S * expf(M - m2) + s2; M = m2; }
      else S += s2 * expf(m2 - M);
    }
    if (t == t0) {
      // the first record is already in rank order
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        if (k >= K) continue;
        const int id = __float_as_int(rec[3 + 2 * k]);
        if (id >= 0) { lv[k] = rec[2 + 2 * k]; li[k] = id; }
      }
      continue;
    }
    // insert each entry by a compare-and-swap pass (fixed indices keep the lists in registers)
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      if (k >= K) continue;
      float cv = rec[2 + 2 * k];
      int ci = __float_as_int(rec[3 + 2 * k]);
      if (ci < 0) continue;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        if (j < K && rank_before(cv, ci, lv[j], li[j])) {
          const float tv = lv[j];
          const int ti = li[j];
          lv[j] = cv; li[j] = ci;
          cv = tv; ci = ti;
        }
      }
    }
  }
}

// Warp reduction of the lanes' sorted lists and (max, sum-exp) pairs (the pairs in a fixed
// butterfly order): lane 0 receives the K best (out_v, out_i) and the combined pair. Each
// round takes the best list head over the lanes and pops it from its owner's list.
EAGLE_DEV void head_merge_warp(int K, float* lv, int* li, float& M, float& S, int lane, float* out_v, int* out_i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, M, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, S, o);
    const float mn = fmaxf(M, m2);
    if (mn != -INFINITY) S = S * expf(M - mn) + s2 * expf(m2 - mn);
    M = mn;
  }
  for (int k = 0; k < K; ++k) {
    float bv;
    int bi;
    const int mine = li[0];
    warp_best(lv[0], li[0], bv, bi);
    if (mine == bi && bi != 0x7fffffff) {
#pragma unroll
      for (int j = 0; j < 15; ++j) { lv[j] = lv[j + 1]; li[j] = li[j + 1]; }
      lv[15] = -INFINITY;
      li[15] = 0x7fffffff;
    }
    if (lane == 0) {
      out_v[k] = bv;
      out_i[k] = bi;
    }
  }
}
