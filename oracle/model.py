"""Oracle model math: Llama-style target and the EAGLE-1 / EAGLE-3 drafters.

Plain numpy, fp64 accumulation. Weights arrive as float32 arrays (an exact
upcast of the stored values). The model rounds to its storage type ("bf16" or
"f32") at fixed points, which are part of the model definition, not of any GPU
code: GEMM inputs (normed activations, attention output, SwiGLU output, the
final-norm feature), the query vector, every KV-cache entry, and every feature
handed to the drafter.

Page references:
- target feature f = input of the LM head, i.e. the final-RMSNorm output; the
  LM head is a single matrix followed by softmax ("EAGLE: Feature-Level
  Drafting", section "The big idea: draft at the feature level"; "EAGLE 三代",
  §2.1);
- EAGLE-1 drafter: embed(tokens) concatenated with features to [.., 2H], an FC
  back to H, one decoder layer, then the shared LM head ("EAGLE 三代", §2.3;
  "EAGLE: Feature-Level Drafting", section "Resolving the uncertainty by feeding
  back the token" for the one-step-advanced token);
- EAGLE-3 drafter: g = FC([l; m; h]) from low/mid/high target layers, combined
  with the token embedding in one decoder layer; on new draft positions the
  drafter's own output a replaces g ("EAGLE 三代", §4.3).

Test infrastructure: only tests, the smoke check and the bench's CPU baseline
use this package.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Dict, List, Optional, Sequence

import numpy as np


def bf16_round(x) -> np.ndarray:
    """Round to the nearest bfloat16 (ties to even), via float32. Returns float64."""
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = a.view(np.uint32).astype(np.uint64)
    u = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) & np.uint64(0xFFFF0000)
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def f32_round(x) -> np.ndarray:
    """Round to float32 and back (a rounding point of the fp32 model)."""
    return np.asarray(x, dtype=np.float32).astype(np.float64)


def no_round(x) -> np.ndarray:
    """No rounding: float64 as is."""
    return np.asarray(x, dtype=np.float64)


def quantizer(dtype: str):
    """Rounding applied at the model's rounding points: bf16, f32, or none ("f64",
    used by tests that compare two exact formulations of the same computation)."""
    return {"bf16": bf16_round, "f32": f32_round, "f64": no_round}[dtype]


def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm of the last axis: x / sqrt(mean(x^2) + eps) * g (Llama-style target layers,
    "EAGLE 三代" page §2.3)."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * g


def silu(x: np.ndarray) -> np.ndarray:
    """SiLU, x * sigmoid(x), the SwiGLU MLP's gate activation."""
    return x / (1.0 + np.exp(-x))


def rope(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotate-half rotary embedding. x [R, heads, d], pos [R] -> rotated copy.
    Pair (i, i + d/2) is rotated by angle pos * theta^(-2i/d)."""
    d = x.shape[-1]
    half = d // 2
    inv = theta ** (-2.0 * np.arange(half, dtype=np.float64) / d)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * inv[None, :]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def logsumexp(v: np.ndarray, axis=-1) -> np.ndarray:
    """log sum exp along `axis`, shifted by the maximum (the softmax normaliser behind each
    draft confidence log c = logit - lse)."""
    mx = np.max(v, axis=axis, keepdims=True)
    return (mx + np.log(np.sum(np.exp(v - mx), axis=axis, keepdims=True))).squeeze(axis)


@dataclass
class KV:
    """One cache: K and V of shape [layers, n_kv, capacity, d], values already rounded."""
    k: np.ndarray
    v: np.ndarray

    @staticmethod
    def empty(layers: int, n_kv: int, cap: int, d: int, dtype: str = "f32") -> "KV":
        """Storage is float32 (exact for bf16/f32 entries); float64 for the unrounded mode."""
        t = np.float64 if dtype == "f64" else np.float32
        return KV(np.zeros((layers, n_kv, cap, d), t), np.zeros((layers, n_kv, cap, d), t))


def attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, visible: np.ndarray) -> np.ndarray:
    """q [R, nq, d]; K, V [n_kv, S, d]; visible bool [R, S] -> [R, nq, d].
    Query head j reads KV head floor(j * n_kv / nq); scale 1/sqrt(d); the softmax
    runs over the visible keys only."""
    R, nq, d = q.shape
    n_kv = K.shape[0]
    grp = nq // n_kv
    Kh = np.repeat(np.asarray(K, np.float64), grp, axis=0)     # [nq, S, d]
    Vh = np.repeat(np.asarray(V, np.float64), grp, axis=0)
    out = np.empty((R, nq, d))
    step = 128
    for r0 in range(0, R, step):
        r1 = min(R, r0 + step)
        s = np.einsum("rhd,hsd->hrs", q[r0:r1], Kh) / np.sqrt(d)
        s = np.where(visible[None, r0:r1, :], s, -np.inf)
        s = s - np.max(s, axis=-1, keepdims=True)
        p = np.exp(s)
        p /= np.sum(p, axis=-1, keepdims=True)
        out[r0:r1] = np.einsum("hrs,hsd->rhd", p, Vh)
    return out


class Layer:
    """One decoder layer's weights (views into the weight dict)."""

    def __init__(self, W: Dict[str, np.ndarray], prefix: str, F: int):
        self.attn_norm = W.get(prefix + "attn_norm")
        self.wqkv = W[prefix + "wqkv"]
        self.wo = W[prefix + "wo"]
        self.mlp_norm = W[prefix + "mlp_norm"]
        self.wg = W[prefix + "wgu"][:F]
        self.wu = W[prefix + "wgu"][F:]
        self.wd = W[prefix + "wd"]
        self.norm_g = W.get(prefix + "norm_g")
        self.norm_e = W.get(prefix + "norm_e")


_UPCAST = {"buf": np.empty(0)}


def mm(a: np.ndarray, w: np.ndarray) -> np.ndarray:
    """a [R, K] (fp64) times w[N, K]^T with fp64 accumulation.

    A float32 w is upcast to float64 exactly, a block of rows at a time into one reused
    buffer (so a large LM head is never copied whole); each output element is the same
    fp64 dot product either way."""
    a = np.asarray(a, np.float64)
    if w.dtype == np.float64:
        return a @ w.T
    N, K = w.shape
    step = max(1, min(N, (1 << 25) // max(K, 1)))     # rows per block: about 256 MB of fp64
    if _UPCAST["buf"].size < step * K:
        _UPCAST["buf"] = np.empty(step * K, np.float64)
    out = np.empty((a.shape[0], N))
    for n0 in range(0, N, step):
        n1 = min(N, n0 + step)
        wb = _UPCAST["buf"][:(n1 - n0) * K].reshape(n1 - n0, K)
        np.copyto(wb, w[n0:n1])
        out[:, n0:n1] = a @ wb.T
    return out


class Model:
    """Target + drafter math over a numpy weight dict laid out as in `synth.weight_specs`."""

    def __init__(self, W: Dict[str, np.ndarray], shape, drafter_kind: int = 1,
                 fuse_layers: Sequence[int] = (0, 0, 0)):
        self.W = W
        self.s = shape
        self.q = quantizer(shape.dtype)
        F = shape.ffn
        self.layers = [Layer(W, f"layers.{i}.", F) for i in range(shape.n_layers)]
        self.drafter_kind = drafter_kind
        self.fuse_layers = tuple(fuse_layers)
        self.dlayer = Layer(W, "draft.", F) if "draft.wqkv" in W else None

    # -- one decoder layer over a set of rows -------------------------------------
    def layer_rows(self, L: Layer, x: np.ndarray, attn_in: np.ndarray, pos: np.ndarray,
                   kv: KV, li: int, slots: np.ndarray, visible: np.ndarray) -> np.ndarray:
        """x: residual stream [R, H]; attn_in: the rounded QKV input [R, K_in].
        Writes this layer's K, V for the rows at `slots`, then every row attends to the
        cache slots marked in `visible` [R, S]. Returns the new residual stream."""
        s, q = self.s, self.q
        nq, nkv, d = s.n_heads, s.n_kv_heads, s.head_dim
        R = x.shape[0]
        qkv = mm(attn_in, L.wqkv)
        qh = qkv[:, :nq * d].reshape(R, nq, d)
        kh = qkv[:, nq * d:(nq + nkv) * d].reshape(R, nkv, d)
        vh = qkv[:, (nq + nkv) * d:].reshape(R, nkv, d)
        qh = q(rope(qh, pos, s.rope_theta))
        kh = q(rope(kh, pos, s.rope_theta))
        vh = q(vh)
        for r in range(R):
            kv.k[li, :, slots[r], :] = kh[r]
            kv.v[li, :, slots[r], :] = vh[r]
        S = visible.shape[1]
        att = attention(qh, kv.k[li, :, :S, :], kv.v[li, :, :S, :], visible)
        h = x + mm(q(att.reshape(R, nq * d)), L.wo)
        n2 = q(rmsnorm(h, L.mlp_norm, s.rms_eps))
        g = mm(n2, L.wg)
        u = mm(n2, L.wu)
        return h + mm(q(silu(g) * u), L.wd)

    # -- target -------------------------------------------------------------------
    def target_rows(self, tokens: np.ndarray, pos: np.ndarray, kv: KV, slots: np.ndarray,
                    visible: np.ndarray):
        """Target forward over rows. Returns (f, captures) where f = rounded final-norm
        output [R, H] (the feature, also the LM-head input) and captures is the list of
        rounded residual-stream outputs of the EAGLE-3 fusion layers (or [])."""
        s, q = self.s, self.q
        x = np.asarray(self.W["embed"][tokens], np.float64)
        caps = {}
        for li, L in enumerate(self.layers):
            n = q(rmsnorm(x, L.attn_norm, s.rms_eps))
            x = self.layer_rows(L, x, n, pos, kv, li, slots, visible)
            if li in self.fuse_layers and self.drafter_kind == 3:
                caps[li] = q(x)
        f = q(rmsnorm(x, self.W["final_norm"], s.rms_eps))
        capl = [caps[i] for i in self.fuse_layers] if self.drafter_kind == 3 else []
        return f, capl

    def logits(self, f: np.ndarray) -> np.ndarray:
        """The shared LM head over features f ("EAGLE: Feature-Level Drafting", "The big idea:
        draft at the feature level": one matrix, then softmax)."""
        return mm(f, self.W["lm_head"])

    # -- drafter ------------------------------------------------------------------
    def fuse(self, caps: List[np.ndarray]) -> np.ndarray:
        """EAGLE-3: g = FC([l; m; h]) (3H -> H), rounded: it is the drafter's feature input."""
        return self.q(mm(np.concatenate(caps, axis=-1), self.W["draft.fc"]))

    def drafter_rows(self, feat: np.ndarray, tokens: np.ndarray, pos: np.ndarray, kv: KV,
                     slots: np.ndarray, visible: np.ndarray) -> np.ndarray:
        """One drafter step over rows. feat: the rounded feature input [R, H] (EAGLE-1: f or the
        parent's predicted feature; EAGLE-3: g or the parent's a); tokens: the one-step-advanced
        token of each row. Returns the rounded drafter output (f-hat or a) [R, H], which feeds
        both the shared LM head and the children's drafter rows."""
        s, q = self.s, self.q
        L = self.dlayer
        e = np.asarray(self.W["embed"][tokens], np.float64)
        if self.drafter_kind == 1:
            z = mm(np.concatenate([e, feat], axis=-1), self.W["draft.fc"])
            attn_in = q(rmsnorm(z, L.attn_norm, s.rms_eps))
            x = z
        else:
            attn_in = np.concatenate([q(rmsnorm(feat, L.norm_g, s.rms_eps)),
                                      q(rmsnorm(e, L.norm_e, s.rms_eps))], axis=-1)
            x = np.asarray(feat, np.float64)
        out = self.layer_rows(L, x, attn_in, pos, kv, 0, slots, visible)
        return q(out)
