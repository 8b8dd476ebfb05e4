"""GPU test helpers (not tests): the oracle's tree policy rerun on the GPU's own node
table, and greedy speculative decoding against the GPU's own plain greedy decoding, bit for
bit."""
import numpy as np
import torch

from eagle_speculative_decoding_cycle_gb300 import _lib as L
from eagle_speculative_decoding_cycle_gb300 import api
from oracle.tree import NodeTable, flatten, rerank, select_expand, static_plan

DEV = "cuda:0"


def gpu_table(eng, b=0):
    tok, par, dep, logv = eng.dump(L.DUMP_NODES)
    t = NodeTable()
    t.token = tok[b].tolist()
    t.parent = par[b].tolist()
    t.depth = dep[b].tolist()
    t.logv = [np.float32(x) for x in logv[b].numpy()]
    return t


def check_tree_policy(eng, wl, b=0):
    """Oracle policy on the GPU's path values reproduces the GPU's expansion, rerank (or, for
    a static tree, the planned rows and kept set), flattening and mask."""
    k, D, m = wl.tree.topk, wl.tree.depth, wl.tree.m
    t = gpu_table(eng, b)
    static = bool(wl.tree.static_parent)
    if static:
        gen, rows = static_plan(wl.tree.static_parent, wl.tree.static_rank, k, D)
    # expansion order: children of the r-th selected depth-d node occupy block r
    for d in range(1, D):
        sel = rows[d] if static else select_expand(NodeTable(t.token, t.parent, t.depth, t.logv), d, k)
        base = k + (d - 1) * k * k
        for r, v in enumerate(sel):
            assert all(t.parent[base + r * k + i] == v for i in range(k))
    st = eng.dump(L.DUMP_STATE)
    ft = flatten(t, sorted(gen) if static else rerank(t, m), int(eng.dump(L.DUMP_TREE)[0][b, 0]))
    tok, pos, par, node, mask = eng.dump(L.DUMP_TREE)
    assert tok[b].tolist() == ft.token.tolist()
    assert par[b].tolist() == ft.parent.tolist()
    assert node[b].tolist() == ft.node.tolist()
    assert np.array_equal(mask[b].numpy().view(np.uint64), ft.mask_words())
    return t, ft, pos[b].numpy()


def spec_vs_plain(wl, weights, prompts, n_new, kv_block=0, max_ctx=None):
    """Greedy speculative decoding against the GPU's own plain greedy decoding of the same
    prompts, bit for bit: the committed tokens must be identical, and so must the top-2
    logit margin of every verify row on an accepted path and the plain step at the same
    position (the margin is a difference of the two largest logits, so equal margins
    mean those logits agree). Returns (accepted rows compared, cycles run)."""
    B = len(prompts)
    D = wl.tree.depth
    T1 = wl.tree.m + 1
    mc = max_ctx or max(len(p) for p in prompts) + 3 * (n_new + D + 2) + 64
    eng = api.Engine(wl, weights, max_batch=B, max_ctx=mc, kv_block=kv_block)
    pd = [p.to(DEV) for p in prompts]
    eng.prefill(pd)
    first = eng.dump(L.DUMP_STATE)["root_tok"][:B].to(torch.int32)
    n_plain = n_new + D + 1
    plain = torch.zeros(B, n_plain, dtype=torch.int32, device=DEV)
    marg = torch.zeros(B, n_plain, dtype=torch.float32, device=DEV)
    eng.decode_plain(n_plain, plain, marg)
    eng.sync()
    gp = torch.cat([first.view(B, 1), plain.cpu()], 1)
    gm = marg.cpu()                                  # gm[b, i]: margin of the logits at token i
    eng.prefill(pd, gp.to(DEV).contiguous())
    got = [[int(first[b])] for b in range(B)]
    out = torch.zeros(B, D + 1, dtype=torch.int32, device=DEV)
    cnt = torch.zeros(B, dtype=torch.int32, device=DEV)
    rows, cycles = 0, 0
    while min(len(x) for x in got) < n_new:
        c0 = [len(x) - 1 for x in got]               # committed index of each root
        eng.cycle(out, cnt)
        eng.sync()
        cycles += 1
        _, val, _, _ = eng.dump(L.DUMP_VERIFY_HEAD)
        acc_len, _, path = eng.dump(L.DUMP_ACCEPT)
        o, c = out.cpu(), cnt.cpu()
        for b in range(B):
            got[b] += o[b, :int(c[b])].tolist()
            acc = [0] + path[b, :int(acc_len[b])].tolist()
            for j, r in enumerate(acc):
                i = c0[b] + j
                if i < n_plain:
                    v = val[b * T1 + r]
                    assert (v[0] - v[1]).item() == gm[b, i].item(), (b, cycles, j, i)
                    rows += 1
    eng.close()
    for b in range(B):
        assert got[b][:n_new] == gp[b, :n_new].tolist(), f"sequence {b} left plain decoding"
    return rows, cycles
