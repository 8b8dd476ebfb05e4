"""Seeded synthetic inputs: workload shapes, random-init weights and prompts.

This module holds only shapes and random draws. It contains none of the
method's arithmetic (no model, no tree policy, no acceptance rule), so that the
CUDA path and the CPU oracle can both take their inputs from it without sharing
any computation.

Workloads follow the model/tree shapes used on the EAGLE pages: a Llama-style
target (decoder layers with RMSNorm, rotary attention and a SwiGLU MLP) whose
frozen embedding and LM head are shared by a one-layer feature drafter
("EAGLE: Feature-Level Drafting", section "The big idea: draft at the feature
level"; "EAGLE 三代", §2.3 and §4.3). All weights are random-init N(0, 0.02),
norm gains are 1, prompts are uniform random token ids.

Weight layout (the layout the C ABI expects, row-major, "out x in"):
  target:  embed [V,H], lm_head [V,H], final_norm [H]
           per layer: attn_norm [H], wqkv [(nq+2nkv)*d, H] = [Wq; Wk; Wv],
           wo [H, nq*d], mlp_norm [H], wgu [2F, H] = [Wgate; Wup], wd [H, F]
  drafter kind 1 (EAGLE-1): fc [H, 2H] over [emb; f], then one target-shaped layer
  drafter kind 3 (EAGLE-3): fc [H, 3H] over [l; m; h], norm_g [H], norm_e [H],
           wqkv [(nq+2nkv)*d, 2H] over [RMSNorm(g); RMSNorm(emb)], wo, mlp_norm, wgu, wd
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Tuple

import torch


@dataclass(frozen=True)
class ModelShape:
    n_layers: int
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    rope_theta: float = 1e4
    rms_eps: float = 1e-5
    dtype: str = "bf16"          # "f32" or "bf16": storage type of weights and KV
    init_std: float = 0.02
    lm_head_std: Optional[float] = None   # defaults to init_std

    @property
    def qkv_out(self) -> int:
        return (self.n_heads + 2 * self.n_kv_heads) * self.head_dim


@dataclass(frozen=True)
class DrafterShape:
    kind: int = 1                              # 1 = EAGLE-1 feature drafter, 3 = EAGLE-3 fused
    fuse_layers: Tuple[int, int, int] = (0, 0, 0)   # EAGLE-3 low/mid/high target layers (0-based)


@dataclass(frozen=True)
class TreeShape:
    topk: int
    depth: int
    m: int
    temperature: float = 0.0       # 0 = greedy
    planted_p: float = 0.0         # probability of planting the reference token per depth
    planted_conf: float = 0.9      # confidence given to a planted token
    # static (EAGLE-1) tree: node i = (parent node or -1 for the root, rank among its
    # parent's drafted children); empty = the EAGLE-2 dynamic tree. m must equal its size.
    static_parent: Tuple[int, ...] = ()
    static_rank: Tuple[int, ...] = ()

    @property
    def n_gen(self) -> int:
        return self.topk + (self.depth - 1) * self.topk * self.topk


@dataclass(frozen=True)
class Workload:
    name: str
    model: ModelShape
    drafter: DrafterShape
    tree: TreeShape
    batch: int
    prompt_len: Tuple[int, int]    # (lo, hi) inclusive; lo == hi for a fixed length
    new_tokens: int
    kv_block: int = 0              # 0 = contiguous KV, else paged block size
    seed: int = 0

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# ---------------------------------------------------------------------------
# The workloads. Shapes follow the Llama-family models the pages measure on.
# ---------------------------------------------------------------------------
TINY = Workload(
    name="tiny-f32-2L-H256-V1024",
    model=ModelShape(n_layers=2, hidden=256, n_heads=4, n_kv_heads=4, head_dim=64, ffn=688,
                     vocab=1024, rope_theta=1e4, dtype="f32"),
    drafter=DrafterShape(kind=1),
    tree=TreeShape(topk=4, depth=4, m=16, temperature=0.0, planted_p=0.8),
    batch=1, prompt_len=(32, 32), new_tokens=64, seed=0)

LLAMA2_7B = Workload(
    name="llama2-7b-eagle1-greedy",
    model=ModelShape(n_layers=32, hidden=4096, n_heads=32, n_kv_heads=32, head_dim=128, ffn=11008,
                     vocab=32000, rope_theta=1e4, dtype="bf16"),
    drafter=DrafterShape(kind=1),
    tree=TreeShape(topk=10, depth=6, m=60, temperature=0.0, planted_p=0.8),
    batch=1, prompt_len=(512, 512), new_tokens=256, seed=0)

LLAMA31_8B_SAMPLE = Workload(
    name="llama3.1-8b-eagle3-t1",
    model=ModelShape(n_layers=32, hidden=4096, n_heads=32, n_kv_heads=8, head_dim=128, ffn=14336,
                     vocab=128256, rope_theta=5e5, dtype="bf16"),
    drafter=DrafterShape(kind=3, fuse_layers=(2, 16, 29)),
    tree=TreeShape(topk=10, depth=8, m=60, temperature=1.0, planted_p=0.8),
    batch=1, prompt_len=(1024, 1024), new_tokens=256, seed=0)

LLAMA_13B_LONG = Workload(
    name="llama-13b-longctx-greedy",
    model=ModelShape(n_layers=40, hidden=5120, n_heads=40, n_kv_heads=40, head_dim=128, ffn=13824,
                     vocab=32000, rope_theta=1e4, dtype="bf16"),
    drafter=DrafterShape(kind=1),
    tree=TreeShape(topk=8, depth=6, m=48, temperature=0.0, planted_p=0.8),
    batch=1, prompt_len=(4096, 4096), new_tokens=512, seed=0)

LLAMA31_8B_BS64 = Workload(
    name="llama3.1-8b-eagle3-bs64-paged",
    model=LLAMA31_8B_SAMPLE.model,
    drafter=DrafterShape(kind=3, fuse_layers=(2, 16, 29)),
    tree=TreeShape(topk=4, depth=5, m=16, temperature=0.0, planted_p=0.8),
    batch=64, prompt_len=(128, 2048), new_tokens=128, kv_block=16, seed=0)

WORKLOADS: Dict[str, Workload] = {w.name: w for w in
                                  (TINY, LLAMA2_7B, LLAMA31_8B_SAMPLE, LLAMA_13B_LONG, LLAMA31_8B_BS64)}

# Small shapes used by tests: several GEMM tiles with ragged tails, both drafter kinds.
SMALL_BF16 = Workload(
    name="small-bf16-3L-H320",
    model=ModelShape(n_layers=3, hidden=320, n_heads=5, n_kv_heads=5, head_dim=64, ffn=832,
                     vocab=1000, rope_theta=1e4, dtype="bf16"),
    drafter=DrafterShape(kind=1),
    tree=TreeShape(topk=5, depth=4, m=12, temperature=0.0, planted_p=0.8),
    batch=1, prompt_len=(40, 40), new_tokens=32, seed=1)

SMALL_BF16_E3 = Workload(
    name="small-bf16-eagle3-gqa",
    model=ModelShape(n_layers=4, hidden=256, n_heads=8, n_kv_heads=2, head_dim=32, ffn=640,
                     vocab=700, rope_theta=5e5, dtype="bf16"),
    drafter=DrafterShape(kind=3, fuse_layers=(0, 1, 3)),
    tree=TreeShape(topk=4, depth=5, m=14, temperature=1.0, planted_p=0.8),
    batch=1, prompt_len=(24, 24), new_tokens=24, seed=2)

# Vocabulary-16 model for exact enumeration of the sampling rule. The LM head uses
# a larger scale so the target distribution is neither flat nor one-hot.
VOCAB16 = Workload(
    name="vocab16-f32",
    model=ModelShape(n_layers=2, hidden=32, n_heads=2, n_kv_heads=2, head_dim=16, ffn=64,
                     vocab=16, rope_theta=1e4, dtype="f32", init_std=0.2, lm_head_std=0.35),
    drafter=DrafterShape(kind=1),
    tree=TreeShape(topk=2, depth=2, m=3, temperature=1.0, planted_p=0.0),
    batch=1, prompt_len=(4, 4), new_tokens=3, seed=3)

# ---------------------------------------------------------------------------
# Seed streams. Sub-stream 0 draws weights, 1 draws prompts. Streams 2.. are the
# counter-based draws the method itself makes (planting, acceptance, Gumbel);
# those are keyed by the workload seed inside each side's Philox generator.
# ---------------------------------------------------------------------------
STREAM_WEIGHTS = 0
STREAM_PROMPTS = 1


def _gen(seed: int, stream: int, device: str) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 16 + stream)
    return g


def weight_specs(model: ModelShape, drafter: Optional[DrafterShape]) -> List[Tuple[str, Tuple[int, ...], float]]:
    """(name, shape, std) in draw order. std 0 means a norm gain (all ones)."""
    H, F, V = model.hidden, model.ffn, model.vocab
    s = model.init_std
    s_lm = model.lm_head_std if model.lm_head_std is not None else s
    specs: List[Tuple[str, Tuple[int, ...], float]] = [
        ("embed", (V, H), s), ("lm_head", (V, H), s_lm), ("final_norm", (H,), 0.0)]
    for i in range(model.n_layers):
        p = f"layers.{i}."
        specs += [(p + "attn_norm", (H,), 0.0), (p + "wqkv", (model.qkv_out, H), s),
                  (p + "wo", (H, model.n_heads * model.head_dim), s), (p + "mlp_norm", (H,), 0.0),
                  (p + "wgu", (2 * F, H), s), (p + "wd", (H, F), s)]
    if drafter is not None:
        p = "draft."
        if drafter.kind == 1:
            specs += [(p + "fc", (H, 2 * H), s), (p + "attn_norm", (H,), 0.0),
                      (p + "wqkv", (model.qkv_out, H), s)]
        else:
            specs += [(p + "fc", (H, 3 * H), s), (p + "norm_g", (H,), 0.0), (p + "norm_e", (H,), 0.0),
                      (p + "wqkv", (model.qkv_out, 2 * H), s)]
        specs += [(p + "wo", (H, model.n_heads * model.head_dim), s), (p + "mlp_norm", (H,), 0.0),
                  (p + "wgu", (2 * F, H), s), (p + "wd", (H, F), s)]
    return specs


def make_weights(w: Workload, device: str = "cpu", with_drafter: bool = True) -> Dict[str, torch.Tensor]:
    """Random-init weights in the storage dtype (float32 or bfloat16) on `device`.

    The values are drawn as float32 N(0, std) by torch's generator on `device` and
    then rounded once to the storage dtype; norm gains are exactly 1.
    """
    dt = torch.float32 if w.model.dtype == "f32" else torch.bfloat16
    g = _gen(w.seed, STREAM_WEIGHTS, device)
    out: Dict[str, torch.Tensor] = {}
    for name, shape, std in weight_specs(w.model, w.drafter if with_drafter else None):
        if std == 0.0:
            out[name] = torch.ones(shape, dtype=dt, device=device)
        else:
            t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
            t.mul_(std)
            out[name] = t.to(dt)
            del t
    return out


def make_prompts(w: Workload) -> List[torch.Tensor]:
    """One int32 tensor of token ids per sequence; lengths uniform in prompt_len."""
    g = _gen(w.seed, STREAM_PROMPTS, "cpu")
    lo, hi = w.prompt_len
    out = []
    for _ in range(w.batch):
        n = lo if lo == hi else int(torch.randint(lo, hi + 1, (1,), generator=g).item())
        out.append(torch.randint(0, w.model.vocab, (n,), generator=g, dtype=torch.int64).to(torch.int32))
    return out


def weights_to_numpy(weights: Dict[str, torch.Tensor]):
    """float32 numpy copies (an exact upcast of bf16 storage)."""
    return {k: v.detach().to("cpu", torch.float32).numpy() for k, v in weights.items()}
