"""Lossless speculative sampling on the GPU: over ~10^6 independent sequences of the
vocabulary-16 model (temperature 1, top-k 2, depth 2, m 3), the joint distribution of the
first three committed tokens (the prefill token and the next two) produced by the
draft-and-verify cycle must match the target's own autoregressive joint (chi-square,
p > 0.001, bins with expected count < 5 merged), as must each position's marginal.
The analytic joint comes from the oracle's plain forward (fp64)."""
import numpy as np
import pytest
import torch
from scipy import stats

from eagle_speculative_decoding_cycle_gb300 import _lib as L
from eagle_speculative_decoding_cycle_gb300 import api, synth
from oracle.cycle import build_model
from oracle.model import KV, logsumexp

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _chi2(obs, exp):
    obs = np.asarray(obs, np.float64).ravel()
    exp = np.asarray(exp, np.float64).ravel()
    big = exp >= 5
    o = np.append(obs[big], obs[~big].sum())
    e = np.append(exp[big], exp[~big].sum())
    if e[-1] < 5:
        o[-2] += o[-1]
        e[-2] += e[-1]
        o, e = o[:-1], e[:-1]
    return stats.chisquare(o, e * o.sum() / e.sum()).pvalue


def test_batched_prefill_matches_single_prefill():
    wl = synth.SMALL_BF16
    weights = {k: v.to(DEV) for k, v in synth.make_weights(wl, "cpu").items()}
    g = torch.Generator().manual_seed(5)
    prompts = [torch.randint(0, wl.model.vocab, (20,), generator=g, dtype=torch.int32) for _ in range(3)]
    eb = api.Engine(wl, weights, max_batch=3)
    eb.prefill([p.to(DEV) for p in prompts])
    st_b = eb.dump(L.DUMP_STATE)
    cand_b = eb.dump(L.DUMP_CAND)
    for i, p in enumerate(prompts):
        es = api.Engine(wl, weights, max_batch=1)
        es.prefill([p.to(DEV)])
        st = es.dump(L.DUMP_STATE)
        ct, cl = es.dump(L.DUMP_CAND)
        assert int(st["root_tok"][0]) == int(st_b["root_tok"][i])
        assert ct[0].tolist() == cand_b[0][i].tolist()
        assert np.allclose(cl[0].numpy(), cand_b[1][i].numpy(), atol=1e-4)
        es.close()
    eb.close()


def test_vocab16_sampling_chi_square():
    wl = synth.VOCAB16
    weights_cpu = synth.make_weights(wl, "cpu")
    weights = {k: v.to(DEV) for k, v in weights_cpu.items()}
    prompt = synth.make_prompts(wl)[0]
    V = wl.model.vocab
    D = wl.tree.depth
    B, runs = 8192, 123
    counts = np.zeros((V, V, V), np.int64)
    accepted = 0
    for run in range(runs):
        eng = api.Engine(wl.replace(seed=1000 + run), weights, max_batch=B, max_ctx=len(prompt) + 4 * (D + 1) + 16)
        eng.prefill([prompt.to(DEV)] * B)
        first = eng.dump(L.DUMP_STATE)["root_tok"].numpy()
        seqs = [[int(t)] for t in first]
        out = torch.zeros(B, D + 1, dtype=torch.int32, device=DEV)
        cnt = torch.zeros(B, dtype=torch.int32, device=DEV)
        for _ in range(2):
            eng.cycle(out, cnt)
            eng.sync()
            o, c = out.cpu().numpy(), cnt.cpu().numpy()
            accepted += int((c > 1).sum())
            for b in range(B):
                seqs[b] += o[b, :c[b]].tolist()
        eng.close()
        t = np.array([s[:3] for s in seqs])
        np.add.at(counts, (t[:, 0], t[:, 1], t[:, 2]), 1)
    # analytic joint P(x0) P(x1 | x0) P(x2 | x0 x1) of the target at T = 1
    M = build_model(synth.weights_to_numpy(weights_cpu), wl)
    s = wl.model

    def cond(seq):
        n = len(seq)
        kv = KV.empty(s.n_layers, s.n_kv_heads, n, s.head_dim)
        p = np.arange(n)
        f, _ = M.target_rows(np.asarray(seq), p, kv, p, np.tril(np.ones((n, n), dtype=bool)))
        lg = M.logits(f[-1:])[0]
        return np.exp(lg - logsumexp(lg))

    base = prompt.tolist()
    joint = np.zeros((V, V, V))
    p0 = cond(base)
    for a in range(V):
        p1 = cond(base + [a])
        for b in range(V):
            joint[a, b] = p0[a] * p1[b] * cond(base + [a, b])
    n = counts.sum()
    assert n == B * runs and accepted > 0
    assert _chi2(counts, joint * n) > 1e-3
    for ax in ((1, 2), (0, 2), (0, 1)):
        assert _chi2(counts.sum(axis=ax), joint.sum(axis=ax) * n) > 1e-3
