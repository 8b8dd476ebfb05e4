"""Oracle of one EAGLE draft-and-verify cycle, plus prefill and plain decoding.

The cycle follows the pages' order ("EAGLE-2: Context-Aware Dynamic Draft
Trees", table "Putting It Together", steps 1-5; "EAGLE: Feature-Level
Drafting", "How EAGLE-2 builds its tree", items 1-4; "EAGLE 三代", §2.3 for the
drafter step and §4.3 for the EAGLE-3 substitution of a for g):

1. the drafter proposes the root's children with confidences;
2. for depth d = 1 .. D-1 the top-k depth-d nodes by path value are expanded in
   one drafter call, each row attending to the drafter context and its own
   expanded ancestors;
3. the global top-m rerank keeps a connected tree, which is flattened with its
   ancestry mask;
4. the target scores the root plus the m kept nodes in one pass with tree
   attention over its KV cache;
5. acceptance (greedy or point-mass rejection) gives the accepted path and the
   bonus token; the accepted rows' KV is compacted and the drafter is advanced
   over the newly committed positions.

Positions: a tree node at depth d sits at target position n + d, n being the
target KV length (the root, the last committed token, is at position n and is
not yet cached). Drafter position p carries (feature of target position p,
embedding of the token at p + 1), the token sequence advanced by one step, so a
node at depth d is expanded at drafter position n + d - 1.

Planted mode is a harness device, not part of the method: given the target's
own plain continuation R, with probability `planted_p` per (sequence, cycle,
depth) the drafter row that extends an on-R prefix gets the next R token
injected as its top-1 with confidence `planted_conf`, by setting that logit to
lse(other logits) + ln(c / (1 - c)). Only the drafter's confidences change.

Test infrastructure: only tests, the smoke check and the bench's CPU baseline
use this package.
"""
from __future__ import annotations

import copy
from dataclasses import dataclass
from typing import Dict, List, Optional, Sequence

import numpy as np

from . import philox
from .accept import argmax_lowest, compact, enumerate_walk, greedy_walk, sample_walk
from .model import KV, Model, logsumexp
from .tree import FlatTree, NodeTable, flatten, rerank, select_expand, static_plan, topk_ids

F32 = np.float32


@dataclass
class Plan:
    table: NodeTable
    flat: FlatTree
    logits: np.ndarray          # target logits [m+1, V] (fp64)
    feats: np.ndarray           # target features of the tree rows [m+1, H] (rounded)
    caps: List[np.ndarray]      # EAGLE-3 captures of the tree rows


class OracleSeq:
    """One sequence's state and its cycle, in plain numpy."""

    def __init__(self, model: Model, wl, seq: int = 0, capacity: Optional[int] = None):
        self.M = model
        self.wl = wl
        self.t = wl.tree
        self.seq = seq
        self.seed = wl.seed
        s = wl.model
        cap = capacity or (wl.prompt_len[1] + wl.new_tokens + 2 * (wl.tree.m + wl.tree.depth) + 8)
        self.cap = cap
        self.kv = KV.empty(s.n_layers, s.n_kv_heads, cap, s.head_dim, s.dtype)
        dcap = cap + wl.tree.depth * wl.tree.topk + 8
        self.dkv = KV.empty(1, s.n_kv_heads, dcap, s.head_dim, s.dtype)
        self.n = 0
        self.committed: List[int] = []
        self.cycle_idx = 0
        self.R: Optional[np.ndarray] = None
        self.on_track = True
        self.root_feat = None
        self.cand_tok: List[int] = []
        self.cand_logc: List[np.float32] = []
        self.accept_lengths: List[int] = []

    # -- helpers ---------------------------------------------------------------
    def _causal_visible(self, n_ctx: int, rows: int) -> np.ndarray:
        S = n_ctx + rows
        vis = np.zeros((rows, S), dtype=bool)
        for r in range(rows):
            vis[r, :n_ctx + r + 1] = True
        return vis

    def _target_pick(self, logits_row: np.ndarray, cycle: int, stream: int, row: int) -> int:
        T = self.t.temperature
        if T == 0.0:
            return argmax_lowest(logits_row)
        g = philox.gumbel_row(self.seed, stream, self.seq, cycle, row, logits_row.shape[0])
        return argmax_lowest(logits_row / T + g)

    def _planted_token(self, path_tokens: Sequence[int]) -> int:
        """R token that a row extending `path_tokens` (tokens below the root) would plant,
        or -1 when planting cannot apply."""
        if self.R is None or self.t.planted_p <= 0.0 or not self.on_track:
            return -1
        c = len(self.committed)
        d = len(path_tokens)
        if c + d >= len(self.R):
            return -1
        if list(path_tokens) != [int(x) for x in self.R[c:c + d]]:
            return -1
        return int(self.R[c + d])

    def _candidates(self, feat_row: np.ndarray, plant_tok: int, cycle: int, depth: int, logits=None):
        """Drafter LM head + softmax + top-k for one row, with planting. Returns (ids, log c fp32).
        `logits`: the row's LM-head output when the caller computed it with other rows."""
        l = self.M.logits(feat_row[None, :])[0] if logits is None else logits
        if plant_tok >= 0:
            u = philox.draw_uniform(self.seed, philox.STREAM_PLANT, self.seq, cycle, depth, 0)
            if F32(u) < F32(self.t.planted_p):
                others = np.delete(l, plant_tok)
                c = self.t.planted_conf
                l = l.copy()
                l[plant_tok] = logsumexp(others) + np.log(c / (1.0 - c))
        logc = l - logsumexp(l)
        ids = topk_ids(l, self.t.topk)
        return [int(i) for i in ids], [F32(logc[i]) for i in ids]

    def _feature_rows(self, f: np.ndarray, caps: List[np.ndarray], rows: Sequence[int]) -> np.ndarray:
        if self.M.drafter_kind == 1:
            return f[list(rows)]
        return self.M.fuse([c[list(rows)] for c in caps])

    # -- prefill ---------------------------------------------------------------
    def prefill(self, prompt: Sequence[int], R: Optional[Sequence[int]] = None, first: Optional[int] = None):
        """Prefill (the EAGLE-2 page, table "Putting It Together", before step 1): the target
        over the prompt gives the first committed token and the features; the drafter runs
        over the prompt positions and its last output gives the root's depth-1 candidates.
        R: the reference continuation for planted mode, or None. first: commit this token
        instead of the oracle's own pick (to replay another implementation's decision in lock
        step, as commit() does for a cycle)."""
        prompt = np.asarray(prompt, dtype=np.int64)
        n = len(prompt)
        self.R = None if R is None else np.asarray(R, dtype=np.int64)
        pos = np.arange(n)
        f, caps = self.M.target_rows(prompt, pos, self.kv, pos, self._causal_visible(0, n))
        self.prefill_logits = self.M.logits(f[-1:])[0]
        if first is None:
            first = self._target_pick(self.prefill_logits, philox.PREFILL_CYCLE, philox.STREAM_GUMBEL, 0)
        self.n = n
        self.committed = [first]
        self.on_track = self.R is None or int(self.R[0]) == first
        feats = self._feature_rows(f, caps, range(n))
        nxt = np.concatenate([prompt[1:], [first]])
        out = self.M.drafter_rows(feats, nxt, pos, self.dkv, pos, self._causal_visible(0, n))
        self.root_feat = out[-1]
        self.cand_tok, self.cand_logc = self._candidates(out[-1], self._planted_token(()), 0, 1)
        return first

    # -- one cycle -------------------------------------------------------------
    def draft_and_verify(self) -> Plan:
        """Steps 1-3 of one cycle: grow the draft tree (EAGLE-2 page, "Path Value Ranks
        Prefixes, Not Isolated Tokens": expand the top-k nodes by path value per depth),
        keep the top-m, flatten with the ancestry mask, and run the target once over the
        tree rows ("The Mask Preserves Tree Semantics in One Target Pass")."""
        t, n = self.t, self.n
        k, D = t.topk, t.depth
        table = NodeTable()
        for tok, lc in zip(self.cand_tok, self.cand_logc):
            table.add(tok, -1, lc)
        feat_of: Dict[int, np.ndarray] = {}
        slot_of: Dict[int, int] = {}
        static = len(t.static_parent) > 0
        if static:
            gen, rows = static_plan(t.static_parent, t.static_rank, k, D)
            if len(gen) != t.m:
                raise ValueError("a static tree must have m nodes")
        for d in range(1, D):
            E = rows[d] if static else select_expand(table, d, k)
            R = len(E)
            feats = np.stack([self.root_feat if table.parent[v] < 0 else feat_of[table.parent[v]] for v in E])
            toks = np.array([table.token[v] for v in E])
            pos = np.full(R, n + d - 1)
            slots = np.array([n + (d - 1) * k + r for r in range(R)])
            for r, v in enumerate(E):
                slot_of[v] = int(slots[r])
            S = n + d * k
            vis = np.zeros((R, S), dtype=bool)
            vis[:, :n] = True
            for r, v in enumerate(E):
                for a in table.path(v):
                    vis[r, slot_of[a]] = True
            out = self.M.drafter_rows(feats, toks, pos, self.dkv, slots, vis)
            lg = self.M.logits(out)       # the shared LM head over all expanded rows at once
            for r, v in enumerate(E):
                feat_of[v] = out[r]
                path_tokens = [table.token[a] for a in table.path(v)]
                ids, lcs = self._candidates(out[r], self._planted_token(path_tokens), self.cycle_idx, d + 1,
                                            logits=lg[r])
                for tok, lc in zip(ids, lcs):
                    table.add(tok, v, lc)
        kept = sorted(gen) if static else rerank(table, t.m)
        return self.verify(table, flatten(table, kept, self.committed[-1]))

    def verify(self, table: NodeTable, flat: FlatTree) -> Plan:
        """Step 3: the target scores the root and the kept nodes of a flattened tree in one
        pass, each row seeing the context and its own ancestors ("EAGLE-2", "The Mask
        Preserves Tree Semantics in One Target Pass"). Also used to verify a tree drafted
        elsewhere (the GPU's, when a near-tie in path values made the two trees differ)."""
        n = self.n
        rows = len(flat.token)
        pos = n + flat.depth
        slots = n + np.arange(rows)
        vis = np.zeros((rows, n + rows), dtype=bool)
        vis[:, :n] = True
        vis[:, n:] = flat.mask
        f, caps = self.M.target_rows(flat.token, pos, self.kv, slots, vis)
        return Plan(table, flat, self.M.logits(f), f, caps)

    def decide(self, plan: Plan):
        """Acceptance on the plan's target logits. Returns (accepted rows, bonus)."""
        T = self.t.temperature
        flat, logits = plan.flat, plan.logits
        if T == 0.0:
            return greedy_walk(flat, [argmax_lowest(r) for r in logits])
        lse = logsumexp(logits / T)
        V = logits.shape[1]

        def p_child(row, tok):
            return float(np.exp(logits[row, tok] / T - lse[row]))

        def uni(row, i):
            return philox.draw_uniform(self.seed, philox.STREAM_ACCEPT, self.seq, self.cycle_idx, i, row)

        def bonus(row, excl):
            g = philox.gumbel_row(self.seed, philox.STREAM_GUMBEL, self.seq, self.cycle_idx, row, V)
            v = logits[row] / T + g
            v[np.asarray(excl, dtype=np.int64)] = -np.inf
            return argmax_lowest(v)

        return sample_walk(flat, p_child, uni, bonus, dtype=np.float64)

    def commit(self, plan: Plan, path: List[int], bonus: int) -> List[int]:
        """Steps 4-5: copy the accepted rows' KV into their final slots, commit the path and
        the bonus token, and run the drafter over the committed rows (features of the root
        and the path) to get the next root's candidates. Returns the committed tokens."""
        n, flat = self.n, plan.flat
        L = len(path)
        compact(self.kv.k, self.kv.v, n, path)
        rows = [0] + list(path)
        new_tokens = [int(flat.token[r]) for r in path] + [int(bonus)]
        feats = self._feature_rows(plan.feats, plan.caps, rows)
        pos = n + np.arange(L + 1)
        vis = self._causal_visible(n, L + 1)
        out = self.M.drafter_rows(feats, np.asarray(new_tokens), pos, self.dkv, pos, vis)
        self.n = n + L + 1
        self.committed += new_tokens
        if self.R is not None:
            c = len(self.committed)
            self.on_track = self.on_track and c <= len(self.R) and \
                [int(x) for x in self.R[:c]] == self.committed
        self.cycle_idx += 1
        self.accept_lengths.append(L)
        self.root_feat = out[-1]
        self.cand_tok, self.cand_logc = self._candidates(out[-1], self._planted_token(()), self.cycle_idx, 1)
        return new_tokens

    def cycle(self) -> List[int]:
        """One draft-and-verify cycle: tree, verify, acceptance walk, commit."""
        plan = self.draft_and_verify()
        path, bonus = self.decide(plan)
        return self.commit(plan, path, bonus)

    def generate(self, new_tokens: int) -> List[int]:
        """Cycles until at least `new_tokens` tokens are committed (the prefill token counts);
        the surplus of the last cycle is dropped."""
        while len(self.committed) < new_tokens:
            self.cycle()
        return self.committed[:new_tokens]

    def outcomes(self, plan: Plan):
        """Exact outcome distribution of the sampling acceptance for this plan."""
        T = self.t.temperature
        p = np.exp(plan.logits / T - logsumexp(plan.logits / T)[:, None])
        return enumerate_walk(plan.flat, p)

    def fork(self) -> "OracleSeq":
        """Independent copy of the sequence state (the model weights are shared)."""
        o = copy.copy(self)
        o.kv = KV(self.kv.k.copy(), self.kv.v.copy())
        o.dkv = KV(self.dkv.k.copy(), self.dkv.v.copy())
        o.committed = list(self.committed)
        o.accept_lengths = list(self.accept_lengths)
        o.cand_tok = list(self.cand_tok)
        o.cand_logc = list(self.cand_logc)
        return o


def plain_decode(model: Model, wl, prompt: Sequence[int], steps: int, seq: int = 0, margins: Optional[list] = None) \
        -> List[int]:
    """Plain autoregressive decoding of the target: the prefill token then `steps - 1`
    one-token passes. Greedy (argmax, lowest id on ties) or Gumbel-argmax sampling.
    If `margins` is a list, the top-2 logit margin of every greedy pick is appended to it."""
    s = wl.model
    prompt = np.asarray(prompt, dtype=np.int64)
    n = len(prompt)
    cap = n + steps + 8
    kv = KV.empty(s.n_layers, s.n_kv_heads, cap, s.head_dim, s.dtype)
    pos = np.arange(n)
    vis = np.tril(np.ones((n, n), dtype=bool))
    f, _ = model.target_rows(prompt, pos, kv, pos, vis)
    T = wl.tree.temperature

    def pick(lrow, cycle, stream):
        if margins is not None:
            top = np.sort(lrow)[-2:]
            margins.append(float(top[1] - top[0]))
        if T == 0.0:
            return argmax_lowest(lrow)
        g = philox.gumbel_row(wl.seed, stream, seq, cycle, 0, lrow.shape[0])
        return argmax_lowest(lrow / T + g)

    out = [pick(model.logits(f[-1:])[0], philox.PREFILL_CYCLE, philox.STREAM_GUMBEL)]
    for step in range(steps - 1):
        p = n + step
        visr = np.ones((1, p + 1), dtype=bool)
        f, _ = model.target_rows(np.array([out[-1]]), np.array([p]), kv, np.array([p]), visr)
        out.append(pick(model.logits(f)[0], step, philox.STREAM_PLAIN))
    return out


def build_model(weights_np: Dict[str, np.ndarray], wl) -> Model:
    """The oracle model of a workload from float32 copies of its weights."""
    return Model(weights_np, wl.model, wl.drafter.kind, wl.drafter.fuse_layers)
