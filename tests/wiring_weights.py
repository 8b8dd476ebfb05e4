"""Constructed drafter weights whose outputs have a closed form (a test helper, not a test).

The drafter's wiring -- which feature and which token feed drafter position p, which
target layers EAGLE-3 fuses, and where the drafter's own output replaces the fused
feature -- is fixed by the pages in words, not by a worked number. These weights make
the drafter an exact identity on one input, so that its candidates can be predicted
from the target alone:

- EAGLE-1 ("EAGLE: Feature-Level Drafting", sections "The big idea: draft at the feature
  level" and "Resolving the uncertainty by feeding back the token"): the FC over
  [emb(x_{p+1}); f_p] keeps one half (`select="feature"` keeps f_p, `select="token"`
  keeps the embedding), and the decoder layer's output projections are zero, so the
  drafter's output at position p is exactly that half. Its candidates are then the top-k
  of the LM head applied to f_p (the target's own next-token distribution at p) or to
  the embedding of the one-step-advanced token x_{p+1}.
- EAGLE-3 ("EAGLE 三代", §4.3): the fusion FC over [l; m; h] keeps one block
  (`select` = 0, 1 or 2), and the attention output projection is zero while the MLP
  stays, so the drafter maps its feature input x to x + MLP(x). The fused g at a
  committed position is then the selected layer's residual-stream output, and a draft
  node's output is that map applied once more than its parent's output, which is the
  drafter's own output a substituted for g.

The final norm gains are drawn away from 1, so that the LM head's input (the final-norm
output) and the pre-norm residual give different logits.
"""
from __future__ import annotations

import dataclasses

import torch

from eagle_speculative_decoding_cycle_gb300 import synth


def eagle3_workload(base: synth.Workload, fuse=(0, 1, 2)) -> synth.Workload:
    """`base` with an EAGLE-3 drafter over the given fusion layers."""
    return base.replace(drafter=synth.DrafterShape(kind=3, fuse_layers=tuple(fuse)))


def constructed(wl: synth.Workload, select, mlp_scale: float = 5.0, seed: int = 7):
    """Weights of `wl` (storage dtype, CPU) with the drafter made an identity on one input.

    EAGLE-1: select in {"feature", "token"}; EAGLE-3: select in {0, 1, 2} (l, m, h)."""
    w = synth.make_weights(wl, "cpu")
    H = wl.model.hidden
    dt = w["draft.fc"].dtype
    fc = torch.zeros(w["draft.fc"].shape, dtype=torch.float32)
    eye = torch.eye(H)
    if wl.drafter.kind == 1:
        if select == "feature":
            fc[:, H:] = eye
        elif select == "token":
            fc[:, :H] = eye
        else:
            raise ValueError(select)
        w["draft.wd"] = torch.zeros_like(w["draft.wd"])
    else:
        j = int(select)
        fc[:, j * H:(j + 1) * H] = eye
        w["draft.wgu"] = (w["draft.wgu"].float() * mlp_scale).to(dt)
        w["draft.wd"] = (w["draft.wd"].float() * mlp_scale).to(dt)
    w["draft.fc"] = fc.to(dt)
    w["draft.wo"] = torch.zeros_like(w["draft.wo"])
    g = torch.Generator().manual_seed(seed)
    w["final_norm"] = (0.5 + torch.rand(H, generator=g)).to(dt)
    return w


def f32_model(wl: synth.Workload) -> synth.Workload:
    """The same shapes stored in fp32 (fast oracle runs on the CPU)."""
    return wl.replace(model=dataclasses.replace(wl.model, dtype="f32"))
