"""The drafter's wiring on the GPU, with the constructed weights of the oracle's wiring pins
(see wiring_weights.py): the drafter reduced to an identity on one input (EAGLE-1: the feature
f_p or the embedding of the token one step ahead; EAGLE-3: one of the fused layers l, m, h,
with its own output substituted for g below the root). After prefill and after every cycle the
GPU's root candidates and their log-confidences must match the oracle's (which the CPU pins tie
to the target alone): ids where the oracle's consecutive confidences are further apart than the
bf16 bound, log-confidences within it. In between, the oracle's tree policy on the GPU's own
node table must reproduce the GPU's tree bit for bit, and the oracle commits the GPU's
decisions."""
import dataclasses

import numpy as np
import pytest
import torch

from eagle_speculative_decoding_cycle_gb300 import _lib as L
from eagle_speculative_decoding_cycle_gb300 import api, synth
from oracle.accept import greedy_walk
from oracle.cycle import OracleSeq, build_model
from spec_plain import check_tree_policy
from wiring_weights import constructed, eagle3_workload

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TOL = 5e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


E1 = synth.SMALL_BF16.replace(tree=synth.TreeShape(topk=4, depth=3, m=10))
_E3 = synth.SMALL_BF16_E3.replace(tree=synth.TreeShape(topk=3, depth=4, m=9))
E3 = eagle3_workload(_E3.replace(model=dataclasses.replace(_E3.model, n_layers=4)), fuse=(0, 1, 2))


def _check_cands(eng, o, k):
    tok, logc = eng.dump(L.DUMP_CAND)
    g_tok, g_lc = tok[0, :k].tolist(), logc[0, :k].double().numpy()
    o_lc = np.asarray(o.cand_logc, np.float64)
    assert np.max(np.abs(g_lc - o_lc)) < TOL, (g_lc, o_lc)
    # the k-th id is left out: its gap to the (k+1)-th, which neither side keeps, is unknown
    for i in range(k - 1):
        apart = (i == 0 or o_lc[i - 1] - o_lc[i] > 2 * TOL) and o_lc[i] - o_lc[i + 1] > 2 * TOL
        if apart:
            assert g_tok[i] == o.cand_tok[i], (i, g_tok, o.cand_tok)


@pytest.mark.parametrize("wl,select", [(E1, "feature"), (E1, "token"), (E3, 0), (E3, 1), (E3, 2)],
                         ids=["eagle1-feature", "eagle1-token", "eagle3-l", "eagle3-m", "eagle3-h"])
def test_gpu_drafter_wiring_matches_the_pinned_oracle(wl, select):
    weights = constructed(wl, select)
    M = build_model(synth.weights_to_numpy(weights), wl)
    prompt = synth.make_prompts(wl)[0]
    eng = api.Engine(wl, {k: v.to(DEV) for k, v in weights.items()})
    eng.prefill([prompt.to(DEV)])
    first = int(eng.dump(L.DUMP_STATE)["root_tok"][0])
    o = OracleSeq(M, wl)
    o.prefill(prompt.numpy(), first=first)
    k, D = wl.tree.topk, wl.tree.depth
    _check_cands(eng, o, k)
    out = torch.zeros(1, D + 1, dtype=torch.int32, device=DEV)
    cnt = torch.zeros(1, dtype=torch.int32, device=DEV)
    for _ in range(3):
        eng.cycle(out, cnt)
        eng.sync()
        t, ft, _ = check_tree_policy(eng, wl)
        hid = eng.dump(L.DUMP_VERIFY_HEAD)[0]
        gp, gb = greedy_walk(ft, hid[:, 0].tolist())
        acc_len, bonus, path = eng.dump(L.DUMP_ACCEPT)
        assert gp == path[0, :int(acc_len[0])].tolist() and gb == int(bonus[0])
        o.commit(o.verify(t, ft), gp, gb)         # the oracle verifies the GPU's tree
        _check_cands(eng, o, k)
    eng.close()
