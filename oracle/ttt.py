"""Oracle of the EAGLE-3 training-time-test (TTT) forward: the multi-step, self-fed drafter
pass with its attention mask, and the per-step token loss. Forward and loss only; no
training.

What the pages fix ("05 · EAGLE 三代" page, section 4.2 "Training-time test", and the
figure of the TTT attention mask after it, Li et al. 2025 Fig. 6): during training the
drafter's own output is fed back for a few more steps, each step is scored by a
cross-entropy on tokens only, the drafter's internal vector is called a (no longer assumed
equal to the target feature), the first step's mask is the ordinary causal one, and from
the second step on each predicted token sees the original sequence plus its own source
chain instead of an ordinary causal prefix. At inference the same page (section 4.3)
feeds a in place of g at new draft positions.

Reading of the indices (the pages give the idea and the mask's shape only):
- a sequence x_0 .. x_{n-1}; the target runs causally over it and g_t is the drafter's
  feature at position t (EAGLE-3: FC([l; m; h]) of the fused layers; EAGLE-1: the
  target feature f_t);
- step 1, sources t = 0 .. n-3: drafter row [g_t; emb(x_{t+1})] at position t, cache
  slot t, seeing slots 0 .. t;
- step s >= 2, sources t = 0 .. n-2-s: drafter row [a_t^(s-1); emb(x_{t+s})] at position
  t+s-1, cache slot n(s-1)+t, seeing the step-1 slots 0 .. t and its own source's
  earlier steps (slots n(j-1)+t, j = 2 .. s);
- the loss of a row is the cross-entropy of x_{t+s+1} under softmax(LM head(a_t^(s)));
  a step's loss is the mean over its rows.
The same steps apply to an EAGLE-1 drafter, whose output is its predicted feature.

Test infrastructure: only tests, the smoke check and the bench's CPU baseline use this
package.
"""
from __future__ import annotations

from typing import List, Tuple

import numpy as np

from .model import KV


def ttt_slot(n: int, s: int, t: int) -> int:
    """Drafter-cache slot of the step-s row of source t."""
    return t if s == 1 else n * (s - 1) + t


def ttt_visible(n: int, s: int, t: int, width: int) -> np.ndarray:
    """Visibility row of the step-s row of source t over `width` slots."""
    v = np.zeros(width, dtype=bool)
    v[:t + 1] = True
    for j in range(2, s + 1):
        v[ttt_slot(n, j, t)] = True
    return v


def cross_entropy(logits: np.ndarray, target: int) -> float:
    """-log softmax(logits)[target], in float64."""
    z = np.asarray(logits, np.float64)
    mx = np.max(z)
    return float(mx + np.log(np.sum(np.exp(z - mx))) - z[target])


def ttt_forward(M, tokens, steps: int) -> Tuple[List[float], List[np.ndarray]]:
    """Losses of steps 1 .. steps and the drafter outputs a^(s) [rows of step s, H]."""
    x = np.asarray(tokens, dtype=np.int64)
    n = len(x)
    if n < steps + 3:
        raise ValueError("sequence too short for this many steps")
    s_ = M.s
    kv = KV.empty(s_.n_layers, s_.n_kv_heads, n, s_.head_dim, s_.dtype)
    pos = np.arange(n)
    vis = np.tril(np.ones((n, n), dtype=bool))
    f, caps = M.target_rows(x, pos, kv, pos, vis)
    g = f if M.drafter_kind == 1 else M.fuse(caps)
    width = n * steps
    dkv = KV.empty(1, s_.n_kv_heads, width, s_.head_dim, s_.dtype)
    losses, outs = [], []
    prev = None
    for s in range(1, steps + 1):
        T = n - 2 if s == 1 else n - 1 - s
        src = np.arange(T)
        feat = g[src] if s == 1 else prev[src]
        toks = x[src + s]
        rpos = src + s - 1
        slots = np.array([ttt_slot(n, s, t) for t in src])
        V = np.stack([ttt_visible(n, s, t, width) for t in src])
        a = M.drafter_rows(feat, toks, rpos, dkv, slots, V)
        lg = M.logits(a)
        rows = [t for t in src if t + s + 1 <= n - 1]
        losses.append(float(np.mean([cross_entropy(lg[t], int(x[t + s + 1])) for t in rows])))
        outs.append(a)
        prev = a
    return losses, outs
