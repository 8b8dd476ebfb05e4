"""Python binding of the EAGLE cycle library: argument marshalling only.

Every step of prefill, the draft-and-verify cycle and plain decoding runs in the CUDA
library (libeagle.so). PyTorch supplies device memory (weights, the workspace, inputs
and outputs) and the CUDA stream.
"""
from __future__ import annotations

import ctypes as C
import dataclasses
from typing import Dict, List, Optional, Sequence

import torch

from . import _lib as L
from .synth import Workload


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def configs(w: Workload, max_batch: Optional[int] = None, max_ctx: Optional[int] = None,
            prefill_chunk: int = 512, kv_block: Optional[int] = None):
    m = w.model
    mc = L.ModelCfg(m.n_layers, m.hidden, m.n_heads, m.n_kv_heads, m.head_dim, m.ffn, m.vocab,
                    m.rope_theta, m.rms_eps, L.DTYPE_F32 if m.dtype == "f32" else L.DTYPE_BF16)
    dc = L.DrafterCfg(w.drafter.kind, (C.c_int * 3)(*w.drafter.fuse_layers))
    t = w.tree
    tc = L.TreeCfg(t.topk, t.depth, t.m, t.temperature, w.seed, t.planted_p, t.planted_conf)
    if max_ctx is None:
        max_ctx = w.prompt_len[1] + w.new_tokens + 4 * (t.depth + 1) + 16
    lim = L.Limits(max_batch or w.batch, max_ctx, w.kv_block if kv_block is None else kv_block, prefill_chunk)
    return mc, dc, tc, lim


def read_stats(stats: torch.Tensor) -> dict:
    """The fields of an eagle_cycle_stats buffer (copied to the host): counters, and each
    phase's device time in microseconds."""
    raw = stats.detach().to("cpu").contiguous().view(torch.uint8)[:L.STATS_BYTES]
    cnt = raw[:24].view(torch.int32).tolist()
    t = raw[24:].view(torch.int64).tolist()
    out = dict(zip(("batch", "active", "accepted", "committed", "max_accepted", "verify_rows"), cnt))
    out["phase_us"] = {p: (t[i + 1] - t[i]) / 1e3 for i, p in enumerate(L.PHASES)}
    out["cycle_us"] = (t[-1] - t[0]) / 1e3
    return out


class Engine:
    """One context of the cycle library over caller-owned torch CUDA tensors."""

    def __init__(self, w: Workload, weights: Dict[str, torch.Tensor], max_batch: Optional[int] = None,
                 max_ctx: Optional[int] = None, prefill_chunk: int = 512,
                 stream: Optional[torch.cuda.Stream] = None, kv_block: Optional[int] = None):
        self.lib = L.lib()
        self.w = w
        self.k_created = w.tree.topk
        self.weights = weights
        self.stream = stream
        self.mc, self.dc, self.tc, self.lim = configs(w, max_batch, max_ctx, prefill_chunk, kv_block)
        nb = self.lib.eagle_workspace_bytes(C.byref(self.mc), C.byref(self.dc), C.byref(self.tc), C.byref(self.lim))
        if nb == 0:
            raise L.EagleError(L.EAGLE_EINVAL, "invalid configuration")
        dev = next(iter(weights.values())).device
        self.workspace = torch.empty(nb, dtype=torch.uint8, device=dev)
        g = lambda n: _ptr(weights.get(n))
        layers = (L.LayerWeights * w.model.n_layers)()
        for i in range(w.model.n_layers):
            p = f"layers.{i}."
            layers[i] = L.LayerWeights(g(p + "attn_norm"), g(p + "wqkv"), g(p + "wo"), g(p + "mlp_norm"),
                                       g(p + "wgu"), g(p + "wd"))
        self._layers = layers
        draft = L.LayerWeights(g("draft.attn_norm"), g("draft.wqkv"), g("draft.wo"), g("draft.mlp_norm"),
                               g("draft.wgu"), g("draft.wd"))
        self.cw = L.Weights(g("embed"), g("lm_head"), g("final_norm"), layers, g("draft.fc"),
                            g("draft.norm_g"), g("draft.norm_e"), draft)
        h = C.c_void_p()
        rc = self.lib.eagle_create(C.byref(self.mc), C.byref(self.dc), C.byref(self.tc), C.byref(self.cw),
                                   C.byref(self.lim), self.workspace.data_ptr(), nb, _stream(stream), C.byref(h))
        L.check(rc, "eagle_create")
        self.h = h
        self.batch = self.lim.max_batch
        if w.tree.static_parent:
            self.set_static_tree(w.tree.static_parent, w.tree.static_rank)
        self._ref = None
        self._tokens = None

    # -- calls ---------------------------------------------------------------------
    def _check(self, rc: int, what: str) -> None:
        if rc != L.EAGLE_OK:
            raise L.EagleError(rc, f"{what}: {self.lib.eagle_last_error(self.h).decode()}")

    def prefill(self, prompts: Sequence[torch.Tensor], ref: Optional[torch.Tensor] = None) -> None:
        """prompts: int32 CUDA tensors, one per sequence. ref: int32 CUDA [B][ref_len] plain
        continuation (first entry = the prefill token) enabling planted mode, or None."""
        self.batch = len(prompts)
        self._tokens = torch.cat([p.to(torch.int32) for p in prompts]).contiguous()
        lens = (C.c_int32 * self.batch)(*[int(p.numel()) for p in prompts])
        self._ref = None if ref is None else ref.to(torch.int32).contiguous()
        rc = self.lib.eagle_prefill(self.h, self.batch, self._tokens.data_ptr(), lens, _ptr(self._ref),
                                    0 if ref is None else int(self._ref.shape[1]))
        self._check(rc, "eagle_prefill")

    def cycle(self, out_tokens: Optional[torch.Tensor] = None, out_count: Optional[torch.Tensor] = None,
              stats: Optional[torch.Tensor] = None) -> None:
        """One cycle. stats (optional): a device tensor from new_stats(), filled by the device
        with the cycle's statistics (parse with read_stats)."""
        if stats is not None and (stats.numel() * stats.element_size() < L.STATS_BYTES or stats.data_ptr() % 8):
            raise ValueError("stats must be an 8-byte aligned device buffer of at least %d bytes" % L.STATS_BYTES)
        self._check(self.lib.eagle_cycle(self.h, _ptr(out_tokens), _ptr(out_count), _ptr(stats)), "eagle_cycle")

    def new_stats(self) -> torch.Tensor:
        """A device buffer for one cycle's statistics."""
        return torch.zeros(L.STATS_BYTES // 8, dtype=torch.int64, device=self.workspace.device)

    def decode_plain(self, n: int, out: torch.Tensor, margin: Optional[torch.Tensor] = None) -> None:
        self._check(self.lib.eagle_decode_plain(self.h, n, _ptr(out), _ptr(margin)), "eagle_decode_plain")

    def set_stop(self, limits: Sequence[int]) -> None:
        """Per-sequence limits on committed tokens (the prefill token included); an empty list
        removes them. A finished sequence is masked out of later cycles."""
        n = len(limits)
        arr = (C.c_int32 * max(n, 1))(*limits)
        self._check(self.lib.eagle_set_stop(self.h, n, arr), "eagle_set_stop")

    def set_tree_budget(self, topk: int, m: int) -> None:
        """Lower the tree's k and m for the next cycles (at most the created values)."""
        self._check(self.lib.eagle_set_tree_budget(self.h, topk, m), "eagle_set_tree_budget")
        self.w = self.w.replace(tree=dataclasses.replace(self.w.tree, topk=topk, m=m))

    def set_graph(self, on: bool) -> None:
        self._check(self.lib.eagle_set_graph(self.h, int(on)), "eagle_set_graph")

    def set_debug(self, flags: int) -> None:
        self._check(self.lib.eagle_set_debug(self.h, flags), "eagle_set_debug")

    def sync(self) -> None:
        """Wait for the stream and raise on latched device errors."""
        self._check(self.lib.eagle_status_sync(self.h), "eagle_status_sync")

    def profile_begin(self, max_launches: int) -> None:
        self._check(self.lib.eagle_profile_begin(self.h, max_launches), "eagle_profile_begin")

    def profile_end(self):
        """(launches, total device ms, total algorithmic bytes) of the profiled GEMM launches."""
        n, ms, by = C.c_int(), C.c_double(), C.c_double()
        self._check(self.lib.eagle_profile_end(self.h, C.byref(n), C.byref(ms), C.byref(by)), "eagle_profile_end")
        return n.value, ms.value, by.value

    def profile_phases(self):
        """(cycles timed, {phase: total device ms}) of the last profiled window."""
        n, ms = C.c_int(), (C.c_double * len(L.PHASES))()
        self._check(self.lib.eagle_profile_phases(self.h, C.byref(n), ms), "eagle_profile_phases")
        return n.value, dict(zip(L.PHASES, list(ms)))

    def profile_verify(self):
        """(verify passes timed, their total device ms) of the last profiled cycles."""
        n, ms = C.c_int(), C.c_double()
        self._check(self.lib.eagle_profile_verify(self.h, C.byref(n), C.byref(ms)), "eagle_profile_verify")
        return n.value, ms.value

    def ttt_forward(self, tokens: torch.Tensor, steps: int) -> torch.Tensor:
        """EAGLE-3 training-time-test forward over one sequence (int32 CUDA tensor): the mean
        token cross-entropy of each of `steps` self-fed drafter steps (float32 CUDA [steps]).
        Reuses sequence 0's caches; prefill again before cycling."""
        x = tokens.to(torch.int32).contiguous()
        loss = torch.zeros(steps, dtype=torch.float32, device=x.device)
        self._check(self.lib.eagle_ttt_forward(self.h, x.data_ptr(), int(x.numel()), steps, loss.data_ptr()),
                    "eagle_ttt_forward")
        return loss

    def set_static_tree(self, parent: Sequence[int], rank: Sequence[int]) -> None:
        """Static (EAGLE-1) tree of len(parent) == m nodes; an empty topology restores the
        dynamic tree."""
        n = len(parent)
        pa = (C.c_int32 * max(n, 1))(*parent)
        ra = (C.c_int32 * max(n, 1))(*rank)
        self._check(self.lib.eagle_set_static_tree(self.h, n, pa, ra), "eagle_set_static_tree")

    def kv_view(self):
        k, v, cap = C.c_void_p(), C.c_void_p(), C.c_int()
        self._check(self.lib.eagle_kv_view(self.h, C.byref(k), C.byref(v), C.byref(cap)), "eagle_kv_view")
        return k.value, v.value, cap.value

    def kv_table(self):
        """Paged target KV: (device pointer of the int32 block table [max_batch][tab_w], tab_w,
        pool blocks per layer, block size)."""
        t, tw, nb, bs = C.c_void_p(), C.c_int(), C.c_int(), C.c_int()
        self._check(self.lib.eagle_kv_table(self.h, C.byref(t), C.byref(tw), C.byref(nb), C.byref(bs)), "eagle_kv_table")
        return t.value, tw.value, nb.value, bs.value

    def dump_raw(self, what: int) -> torch.Tensor:
        n = self.lib.eagle_dump_bytes(self.h, what)
        buf = torch.empty(n, dtype=torch.uint8, device=self.workspace.device)
        self._check(self.lib.eagle_debug_dump(self.h, what, buf.data_ptr(), n), "eagle_debug_dump")
        return buf

    def dump(self, what: int):
        """Parsed debug view (host tensors)."""
        B = self.batch
        t = self.w.tree
        k, D, T1 = t.topk, t.depth, t.m + 1
        NG = t.n_gen
        raw = self.dump_raw(what).cpu()
        i32 = lambda a, b: raw[a:b].view(torch.int32)
        f32 = lambda a, b: raw[a:b].view(torch.float32)
        if what == L.DUMP_STATE:
            s = i32(0, 7 * B * 4).view(7, B)
            return dict(zip(["ctx_len", "root_tok", "committed", "on_track", "cycle", "acc_len", "bonus"], s))
        if what == L.DUMP_CAND:
            kc = self.k_created
            return i32(0, B * kc * 4).view(B, kc), f32(B * kc * 4, 2 * B * kc * 4).view(B, kc)
        if what == L.DUMP_NODES:
            n = B * NG * 4
            return (i32(0, n).view(B, NG), i32(n, 2 * n).view(B, NG), i32(2 * n, 3 * n).view(B, NG),
                    f32(3 * n, 4 * n).view(B, NG))
        if what == L.DUMP_TREE:
            n = B * T1 * 4
            W = (T1 + 63) // 64
            mask = raw[4 * n:4 * n + B * T1 * W * 8].view(torch.int64).view(B, T1, W)
            return (i32(0, n).view(B, T1), i32(n, 2 * n).view(B, T1), i32(2 * n, 3 * n).view(B, T1),
                    i32(3 * n, 4 * n).view(B, T1), mask)
        if what == L.DUMP_ACCEPT:
            return i32(0, B * 4), i32(B * 4, 2 * B * 4), i32(2 * B * 4, (2 * B + B * D) * 4).view(B, D)
        if what == L.DUMP_VERIFY_HEAD:
            K = 1 if t.temperature > 0 else 2
            R = B * T1
            a = R * K * 4
            return (i32(0, a).view(R, K), f32(a, 2 * a).view(R, K), f32(2 * a, 2 * a + R * 4),
                    f32(2 * a + R * 4, 2 * a + R * 4 + R * k * 4).view(R, k))
        if what == L.DUMP_VERIFY_LOGITS:
            return f32(0, raw.numel()).view(B * T1, self.w.model.vocab)
        if what == L.DUMP_FEATURES:
            dt = torch.float32 if self.w.model.dtype == "f32" else torch.bfloat16
            return raw.view(dt).view(B * T1, self.w.model.hidden)
        if what == L.DUMP_TTT:
            H = self.w.model.hidden
            es = 4 if self.w.model.dtype == "f32" else 2
            R = raw.numel() // (H * es + 4)
            dt = torch.float32 if es == 4 else torch.bfloat16
            return raw[:R * H * es].view(dt).view(R, H), f32(R * H * es, raw.numel())
        raise ValueError(what)

    def close(self) -> None:
        if getattr(self, "h", None):
            self.lib.eagle_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ---- kernel-level entry points ----------------------------------------------------------------
def _dtype_code(t: torch.Tensor) -> int:
    return L.DTYPE_F32 if t.dtype == torch.float32 else L.DTYPE_BF16


def gemm(W: torch.Tensor, X: torch.Tensor, epi: int = 0, out: Optional[torch.Tensor] = None,
         stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Y = X W^T through the library's GEMM (tcgen05 for bf16, FFMA for fp32)."""
    lib = L.lib()
    N, K = W.shape
    M = X.shape[0]
    if epi == 4:            # SwiGLU: W holds [gate; up], the output has half as many features
        N //= 2
    if out is None:
        out = torch.zeros(M, N, dtype=torch.bfloat16 if epi in (1, 4) else torch.float32, device=X.device)
    nb = lib.eagle_op_gemm_scratch_bytes(M, 2 * N if epi == 4 else N)
    scratch = torch.zeros(max(nb, 1), dtype=torch.uint8, device=X.device)
    rc = lib.eagle_op_gemm(_dtype_code(W), _stream(stream), W.data_ptr(), N, K, X.data_ptr(), M, epi,
                           out.data_ptr(), out.stride(0), scratch.data_ptr(), nb)
    L.check(rc, "eagle_op_gemm")
    return out


def lm_head(W: torch.Tensor, X: torch.Tensor, K: int, inv_t: float = 1.0, gumbel: bool = False,
            lse_excl: bool = False, specials: Optional[torch.Tensor] = None,
            row_seq: Optional[torch.Tensor] = None, row_key: Optional[torch.Tensor] = None,
            cycle: int = 0, seed: int = 0, stream_id: int = 4,
            stream: Optional[torch.cuda.Stream] = None):
    """Fused LM head: returns (top_id [M][K], top_val [M][K], lse [M], spec_logit [M][S] or None)."""
    lib = L.lib()
    V, H = W.shape
    M = X.shape[0]
    dev = X.device
    dt = _dtype_code(W)
    nb = lib.eagle_op_lm_head_scratch_bytes(dt, V, M, K)
    scratch = torch.zeros(nb, dtype=torch.uint8, device=dev)
    top_id = torch.empty(M, K, dtype=torch.int32, device=dev)
    top_val = torch.empty(M, K, dtype=torch.float32, device=dev)
    lse = torch.empty(M, dtype=torch.float32, device=dev)
    S = 0 if specials is None else specials.shape[1]
    spec_logit = None if specials is None else torch.full((M, S), float("nan"), device=dev)
    rc = lib.eagle_op_lm_head(dt, _stream(stream), W.data_ptr(), V, H, X.data_ptr(), M, K, inv_t, int(gumbel),
                              int(lse_excl), _ptr(specials), S, _ptr(spec_logit), _ptr(row_seq), _ptr(row_key),
                              cycle, seed, stream_id, top_id.data_ptr(), top_val.data_ptr(), lse.data_ptr(),
                              scratch.data_ptr(), nb)
    L.check(rc, "eagle_op_lm_head")
    return top_id, top_val, lse, spec_logit


def attention(q, kcache, vcache, row_seq, row_slot, ctx_len, rows_per_seq, mode, tree_T=0, mask=None,
              scale=0.0, split_kv: bool = True, stream: Optional[torch.cuda.Stream] = None,
              max_batch: Optional[int] = None) -> torch.Tensor:
    """q [R][nq][d]; caches [B][nkv][cap][d]; returns out [R][nq][d]. max_batch: the caches'
    sequences B (default), which also sets the key-split length of an engine of that batch."""
    lib = L.lib()
    R, nq, d = q.shape
    _, nkv, cap, _ = kcache.shape
    out = torch.empty_like(q)
    mw = 0 if mask is None else mask.shape[1]
    nb = lib.eagle_op_attention_scratch_bytes(R, nq, d) if split_kv else 0
    scratch = torch.empty(max(nb, 1), dtype=torch.uint8, device=q.device)
    rc = lib.eagle_op_attention(_dtype_code(q), _stream(stream), q.data_ptr(), kcache.data_ptr(), vcache.data_ptr(),
                                out.data_ptr(), R, nq, nkv, d, cap, rows_per_seq, row_seq.data_ptr(),
                                row_slot.data_ptr(), ctx_len.data_ptr(), mode, tree_T, _ptr(mask), mw, scale,
                                int(kcache.shape[0]) if max_batch is None else max_batch,
                                scratch.data_ptr() if nb else None, nb)
    L.check(rc, "eagle_op_attention")
    return out


def tree_build(k: int, depth: int, m: int, cand_tok, cand_logc, child_tok, child_logc, ctx_len, root_tok,
               stream: Optional[torch.cuda.Stream] = None):
    """Injected-confidence tree growth + rerank. Returns dict of node and tree tensors."""
    lib = L.lib()
    B = cand_tok.shape[0]
    dev = cand_tok.device
    NG = k + (depth - 1) * k * k
    T1 = m + 1
    W = (T1 + 63) // 64
    o = {n: torch.empty(B, NG, dtype=torch.int32, device=dev) for n in ("node_tok", "node_parent", "node_depth")}
    o["node_logv"] = torch.empty(B, NG, dtype=torch.float32, device=dev)
    for n in ("tree_tok", "tree_pos", "tree_parent", "tree_node"):
        o[n] = torch.empty(B, T1, dtype=torch.int32, device=dev)
    o["tree_mask"] = torch.empty(B, T1, W, dtype=torch.int64, device=dev)
    nb = lib.eagle_op_tree_scratch_bytes(B, k, depth, m)
    scratch = torch.zeros(nb, dtype=torch.uint8, device=dev)
    rc = lib.eagle_op_tree_build(_stream(stream), B, k, depth, m, cand_tok.data_ptr(), cand_logc.data_ptr(),
                                 _ptr(child_tok), _ptr(child_logc), ctx_len.data_ptr(), root_tok.data_ptr(),
                                 o["node_tok"].data_ptr(), o["node_parent"].data_ptr(), o["node_depth"].data_ptr(),
                                 o["node_logv"].data_ptr(), o["tree_tok"].data_ptr(), o["tree_pos"].data_ptr(),
                                 o["tree_parent"].data_ptr(), o["tree_node"].data_ptr(), o["tree_mask"].data_ptr(),
                                 scratch.data_ptr(), nb)
    L.check(rc, "eagle_op_tree_build")
    return o


def compact(kcache, vcache, n_old, acc_len, acc_path, stream: Optional[torch.cuda.Stream] = None) -> None:
    """In-place KV compaction; caches [layers][B][nkv][cap][d]."""
    lib = L.lib()
    layers, B, nkv, cap, d = kcache.shape
    rc = lib.eagle_op_compact(_dtype_code(kcache), _stream(stream), kcache.data_ptr(), vcache.data_ptr(), layers, B,
                              nkv, cap, d, n_old.data_ptr(), acc_len.data_ptr(), acc_path.data_ptr(),
                              acc_path.shape[1])
    L.check(rc, "eagle_op_compact")


def plan_budget(candidates, rows_pts: Sequence[int], verify_us: Sequence[float], batch: int):
    """Batch-aware draft budget (eagle_plan_budget). candidates: list of (k, draft_us,
    exp_tokens) with exp_tokens[m-1] the expected committed tokens of an m-node tree.
    Returns (k, m, tokens per microsecond)."""
    lib = L.lib()
    n_k = len(candidates)
    ks = (C.c_int32 * n_k)(*[c[0] for c in candidates])
    dr = (C.c_float * n_k)(*[c[1] for c in candidates])
    mm = (C.c_int32 * n_k)(*[len(c[2]) for c in candidates])
    flat = [float(v) for c in candidates for v in c[2]]
    ex = (C.c_float * max(1, len(flat)))(*flat)
    rp = (C.c_int32 * len(rows_pts))(*rows_pts)
    vu = (C.c_float * len(verify_us))(*verify_us)
    bk, bm, rate = C.c_int32(), C.c_int32(), C.c_float()
    L.check(lib.eagle_plan_budget(n_k, ks, dr, mm, ex, len(rows_pts), rp, vu, batch, C.byref(bk), C.byref(bm),
                                  C.byref(rate)), "eagle_plan_budget")
    return bk.value, bm.value, rate.value
