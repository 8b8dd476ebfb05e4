"""GPU test helper (not a test): greedy speculative decoding against the GPU's own plain
greedy decoding, bit for bit."""
import torch

from eagle_speculative_decoding_cycle_gb300 import _lib as L
from eagle_speculative_decoding_cycle_gb300 import api

DEV = "cuda:0"


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
