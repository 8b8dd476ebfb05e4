"""GPU kernel-level parity against the CPU oracle, through the C ABI (eagle_ops.h).

Float tolerances follow the arithmetic: the GEMMs multiply bf16 (or fp32) inputs exactly
and accumulate in fp32, so an output differs from the fp64 oracle by a few fp32 roundings
of partial sums no larger than sum_k |x_k w_k|; we allow 1e-5 * sum_k |x_k w_k| per
element (about 170 fp32 ulps of that sum), while a dropped 64-wide k-block or a wrong
tile moves an output by about 8/K of it (2e-3 at K = 4096). Index work is compared bit
for bit on the same inputs."""
import numpy as np
import pytest
import torch

from eagle_speculative_decoding_cycle_gb300 import api
from oracle.accept import compact as oracle_compact
from oracle.model import attention as oracle_attention
from oracle.model import logsumexp
from oracle.tree import NodeTable, flatten, rerank, select_expand, topk_ids

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


GEMM_TOL = 1e-5


def _rand(shape, g, dtype, scale=1.0):
    return (torch.randn(shape, generator=g) * scale).to(dtype)


def _ref_mm(X, W):
    x = X.double().numpy()
    w = W.double().numpy()
    return x @ w.T, np.abs(x) @ np.abs(w).T


GEMM_SHAPES = [(1, 128, 64), (7, 300, 200), (61, 640, 320), (61, 12288 // 4, 4096 // 4), (16, 1000, 256),
               (17, 4096, 1024), (100, 257, 136), (200, 384, 512), (300, 520, 264), (61, 4096, 11008),
               # several 256-row token tiles: the CTAs split into one slice per token tile
               (1088, 1536, 1024), (600, 4096, 4096), (1300, 640, 2048), (1025, 384, 520)]


@pytest.mark.parametrize("M,N,K", GEMM_SHAPES)
def test_gemm_bf16_matches_oracle(M, N, K):
    g = torch.Generator().manual_seed(M * 7919 + N * 31 + K)
    X = _rand((M, K), g, torch.bfloat16)
    W = _rand((N, K), g, torch.bfloat16, 0.05)
    Y = api.gemm(W.to(DEV), X.to(DEV), epi=0).cpu().double().numpy()
    ref, mag = _ref_mm(X, W)
    assert np.all(np.abs(Y - ref) <= GEMM_TOL * mag + 1e-6), np.max(np.abs(Y - ref) / (mag + 1e-9))


@pytest.mark.parametrize("M,N,K", [(61, 640, 320), (5, 4096, 4096), (130, 520, 264), (700, 512, 768)])
def test_gemm_bf16_epilogues(M, N, K):
    g = torch.Generator().manual_seed(11)
    X = _rand((M, K), g, torch.bfloat16)
    W = _rand((N, K), g, torch.bfloat16, 0.05)
    ref, mag = _ref_mm(X, W)
    yb = api.gemm(W.to(DEV), X.to(DEV), epi=1).cpu().double().numpy()
    assert np.all(np.abs(yb - ref) <= GEMM_TOL * mag + np.abs(ref) * 2.0 ** -8 + 1e-6)
    base = torch.randn(M, N, generator=g)
    acc = base.clone().to(DEV)
    api.gemm(W.to(DEV), X.to(DEV), epi=2, out=acc)
    assert np.all(np.abs(acc.cpu().double().numpy() - (base.double().numpy() + ref)) <= GEMM_TOL * mag + 1e-5)


def test_gemm_bf16_repeatable():
    """Stream-K split tiles are summed in a fixed order: bitwise identical reruns."""
    g = torch.Generator().manual_seed(3)
    X = _rand((61, 4096), g, torch.bfloat16).to(DEV)
    W = _rand((4096, 4096), g, torch.bfloat16, 0.02).to(DEV)
    a = api.gemm(W, X)
    b = api.gemm(W, X)
    assert torch.equal(a, b)


@pytest.mark.parametrize("M,N,K", [(1, 64, 32), (17, 1024, 256), (33, 700, 96)])
def test_gemm_f32_matches_oracle(M, N, K):
    g = torch.Generator().manual_seed(5)
    X = torch.randn(M, K, generator=g)
    W = torch.randn(N, K, generator=g) * 0.05
    Y = api.gemm(W.to(DEV), X.to(DEV)).cpu().double().numpy()
    ref, mag = _ref_mm(X, W)
    assert np.all(np.abs(Y - ref) <= 1e-5 * mag + 1e-7)


@pytest.mark.parametrize("dtype,V,H,M,K", [(torch.bfloat16, 32000, 512, 61, 2), (torch.bfloat16, 1000, 320, 10, 5),
                                           (torch.float32, 1024, 256, 17, 4), (torch.bfloat16, 5000, 256, 3, 10),
                                           # several 256-row token tiles, the largest K, a ragged last tile
                                           (torch.bfloat16, 3000, 256, 300, 16), (torch.bfloat16, 2056, 512, 600, 3)])
def test_lm_head_topk_and_lse(dtype, V, H, M, K):
    """Fused head vs the oracle's top-k / log-sum-exp on the same logits (the GPU GEMM's
    own fp32 logits, so index results must agree bit for bit)."""
    g = torch.Generator().manual_seed(V + M)
    X = _rand((M, H), g, dtype).to(DEV)
    W = _rand((V, H), g, dtype, 0.05).to(DEV)
    logits = api.gemm(W, X).cpu().double().numpy()
    ids, vals, lse, _ = api.lm_head(W, X, K)
    ids, vals, lse = ids.cpu().numpy(), vals.cpu().numpy(), lse.cpu().numpy()
    for r in range(M):
        want = topk_ids(logits[r].astype(np.float32), K)
        assert list(ids[r]) == list(want)
        assert np.array_equal(vals[r], logits[r][want].astype(np.float32))
        assert abs(lse[r] - logsumexp(logits[r])) < 1e-4


@pytest.mark.parametrize("M,K", [(7, 8), (260, 16)])
def test_lm_head_equal_logits_rank_by_id(M, K):
    """Vocabulary rows repeat every 50 ids, so every logit value occurs 20 times across
    tiles and quarters of a tile: the kept entries must be the lowest ids of the best
    values, in value then id order (the oracle's top-k rule)."""
    g = torch.Generator().manual_seed(21)
    V, H = 1000, 256
    X = _rand((M, H), g, torch.bfloat16).to(DEV)
    W = _rand((50, H), g, torch.bfloat16, 0.05).repeat(V // 50, 1).contiguous().to(DEV)
    logits = api.gemm(W, X).cpu().double().numpy()
    ids, vals, lse, _ = api.lm_head(W, X, K)
    ids, lse = ids.cpu().numpy(), lse.cpu().numpy()
    for r in range(M):
        want = topk_ids(logits[r].astype(np.float32), K)
        assert list(ids[r]) == list(want)
        assert abs(lse[r] - logsumexp(logits[r])) < 1e-4


def test_lm_head_specials_and_gumbel():
    """Specials are left out of ranking (and of the lse when asked) and their logits are
    reported; Gumbel ranking equals the oracle's Philox-keyed Gumbel-argmax."""
    from oracle import philox
    g = torch.Generator().manual_seed(9)
    V, H, M, S = 3000, 256, 6, 3
    X = _rand((M, H), g, torch.bfloat16).to(DEV)
    W = _rand((V, H), g, torch.bfloat16, 0.08).to(DEV)
    logits = api.gemm(W, X).cpu().double().numpy()
    spec = torch.tensor([[int(np.argmax(logits[r])), 5 + r, -1] for r in range(M)], dtype=torch.int32)
    seq = torch.tensor([2] * M, dtype=torch.int32)
    key = torch.arange(M, dtype=torch.int32)
    T = 0.7
    ids, vals, lse, sl = api.lm_head(W, X, 1, inv_t=1 / T, gumbel=True, lse_excl=False, specials=spec.to(DEV),
                                     row_seq=seq.to(DEV), row_key=key.to(DEV), cycle=13, seed=1234,
                                     stream_id=philox.STREAM_GUMBEL)
    ids, lse, sl = ids.cpu().numpy(), lse.cpu().numpy(), sl.cpu().numpy()
    for r in range(M):
        lr = logits[r].astype(np.float32).astype(np.float64)
        gmb = philox.gumbel_row(1234, philox.STREAM_GUMBEL, 2, 13, r, V)
        v = lr * np.float32(1 / T) + gmb
        v[[s for s in spec[r].tolist() if s >= 0]] = -np.inf
        assert ids[r, 0] == int(np.argmax(v))
        assert abs(lse[r] - logsumexp(lr / T)) < 1e-3
        assert sl[r, 0] == np.float32(logits[r][spec[r, 0]])
        assert sl[r, 1] == np.float32(logits[r][spec[r, 1]])
    ids2, _, lse2, _ = api.lm_head(W, X, 2, lse_excl=True, specials=spec.to(DEV))
    for r in range(M):
        lr = logits[r].copy()
        ex = [s for s in spec[r].tolist() if s >= 0]
        assert list(ids2[r].cpu().numpy()) == list(topk_ids(lr.astype(np.float32), 2, exclude=ex))
        assert abs(float(lse2[r]) - logsumexp(np.delete(lr, ex))) < 1e-4


def _mask_words(mask):
    n = mask.shape[0]
    W = (mask.shape[1] + 63) // 64
    out = np.zeros((n, W), dtype=np.uint64)
    for i in range(n):
        for j in np.flatnonzero(mask[i]):
            out[i, j // 64] |= np.uint64(1) << np.uint64(j % 64)
    return torch.from_numpy(out.view(np.int64))


@pytest.mark.parametrize("dtype,nq,nkv,d,B,T,ctx", [(torch.float32, 4, 4, 64, 1, 17, 40),
                                                     (torch.bfloat16, 8, 2, 32, 2, 70, 33),
                                                     (torch.bfloat16, 32, 8, 128, 1, 61, 300),
                                                     (torch.bfloat16, 5, 5, 64, 3, 13, 0)])
def test_tree_attention_matches_oracle(dtype, nq, nkv, d, B, T, ctx):
    g = torch.Generator().manual_seed(nq * 100 + T)
    rng = np.random.default_rng(T)
    cap = ctx + T + 5
    kc = _rand((B, nkv, cap, d), g, dtype)
    vc = _rand((B, nkv, cap, d), g, dtype)
    q = _rand((B * T, nq, d), g, dtype)
    masks = []
    for b in range(B):
        parent = [-1] + [int(rng.integers(0, i)) for i in range(1, T)]
        m = np.zeros((T, T), dtype=bool)
        for i in range(T):
            a = i
            while a >= 0:
                m[i, a] = True
                a = parent[a]
        masks.append(m)
    mask = torch.cat([_mask_words(m) for m in masks])
    ctx_len = torch.full((B,), ctx, dtype=torch.int32)
    row_seq = torch.repeat_interleave(torch.arange(B, dtype=torch.int32), T)
    row_slot = (ctx + torch.arange(T, dtype=torch.int32)).repeat(B)
    out = api.attention(q.to(DEV), kc.to(DEV), vc.to(DEV), row_seq.to(DEV), row_slot.to(DEV), ctx_len.to(DEV), T, 1,
                        T, mask.to(DEV)).cpu().double().numpy()
    tol = 1e-5 if dtype == torch.float32 else 2e-2
    for b in range(B):
        vis = np.zeros((T, ctx + T), dtype=bool)
        vis[:, :ctx] = True
        vis[:, ctx:] = masks[b]
        want = oracle_attention(q[b * T:(b + 1) * T].double().numpy(), kc[b, :, :ctx + T].double().numpy(),
                                vc[b, :, :ctx + T].double().numpy(), vis)
        assert np.max(np.abs(out[b * T:(b + 1) * T] - want)) < tol


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_causal_attention_matches_oracle(dtype):
    g = torch.Generator().manual_seed(2)
    nq, nkv, d, R, cap = 4, 2, 64, 77, 90
    kc = _rand((1, nkv, cap, d), g, dtype)
    vc = _rand((1, nkv, cap, d), g, dtype)
    q = _rand((R, nq, d), g, dtype)
    ctx = 5
    row_slot = ctx + torch.arange(R, dtype=torch.int32)
    out = api.attention(q.to(DEV), kc.to(DEV), vc.to(DEV), torch.zeros(R, dtype=torch.int32, device=DEV),
                        row_slot.to(DEV), torch.zeros(1, dtype=torch.int32, device=DEV), R, 0).cpu().double().numpy()
    S = ctx + R
    vis = np.zeros((R, S), dtype=bool)
    for r in range(R):
        vis[r, :ctx + r + 1] = True
    want = oracle_attention(q.double().numpy(), kc[0, :, :S].double().numpy(), vc[0, :, :S].double().numpy(), vis)
    assert np.max(np.abs(out - want)) < (1e-5 if dtype == torch.float32 else 2e-2)


def _oracle_tree(k, D, m, cand_tok, cand_logc, child_tok, child_logc, root, ctx):
    t = NodeTable()
    for i in range(k):
        t.add(int(cand_tok[i]), -1, np.float32(cand_logc[i]))
    for d in range(1, D):
        for r, v in enumerate(select_expand(t, d, k)):
            for i in range(k):
                t.add(int(child_tok[d - 1, r, i]), v, np.float32(child_logc[d - 1, r, i]))
    kept = rerank(t, m)
    return t, flatten(t, kept, root)


@pytest.mark.parametrize("k,D,m,ties", [(4, 4, 16, False), (10, 6, 60, False), (10, 8, 60, True), (2, 3, 5, True),
                                        (4, 5, 16, True), (8, 6, 48, False), (1, 4, 4, False), (3, 1, 2, False)])
def test_tree_build_bit_exact(k, D, m, ties):
    rng = np.random.default_rng(k * 100 + D * 10 + m)
    B = 3
    pool = np.log(np.array([1.0, 0.5, 0.25, 0.9, 0.0625], np.float32))

    def lc(shape):
        if ties:
            return pool[rng.integers(0, len(pool), size=shape)].astype(np.float32)
        return np.log(rng.uniform(1e-5, 1.0, size=shape)).astype(np.float32)

    cand_tok = np.stack([rng.choice(1000, k, replace=False) for _ in range(B)]).astype(np.int32)
    cand_logc = lc((B, k))
    child_tok = rng.integers(0, 1000, size=(B, max(D - 1, 1), k, k)).astype(np.int32)
    child_logc = lc((B, max(D - 1, 1), k, k))
    ctx = np.array([5, 100, 7], dtype=np.int32)
    root = np.array([11, 22, 33], dtype=np.int32)
    T = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    o = api.tree_build(k, D, m, T(cand_tok), T(cand_logc), T(child_tok), T(child_logc), T(ctx), T(root))
    o = {n: v.cpu().numpy() for n, v in o.items()}
    for b in range(B):
        t, ft = _oracle_tree(k, D, m, cand_tok[b], cand_logc[b], child_tok[b], child_logc[b], root[b], ctx[b])
        NG = len(t)
        assert list(o["node_tok"][b][:NG]) == t.token
        assert list(o["node_parent"][b][:NG]) == t.parent
        assert list(o["node_depth"][b][:NG]) == t.depth
        assert np.array_equal(o["node_logv"][b][:NG], np.array(t.logv, np.float32))
        assert list(o["tree_tok"][b]) == list(ft.token)
        assert list(o["tree_parent"][b]) == list(ft.parent)
        assert list(o["tree_node"][b]) == list(ft.node)
        assert list(o["tree_pos"][b]) == list(ctx[b] + ft.depth)
        assert np.array_equal(o["tree_mask"][b].view(np.uint64), ft.mask_words())


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_compaction_bit_exact(dtype):
    g = torch.Generator().manual_seed(4)
    layers, B, nkv, cap, d = 3, 2, 4, 40, 64
    kc = _rand((layers, B, nkv, cap, d), g, dtype)
    vc = _rand((layers, B, nkv, cap, d), g, dtype)
    n_old = torch.tensor([10, 3], dtype=torch.int32)
    acc_len = torch.tensor([3, 0], dtype=torch.int32)
    acc_path = torch.tensor([[2, 5, 9, 0, 0, 0], [0, 0, 0, 0, 0, 0]], dtype=torch.int32)
    k_ref = kc.float().numpy().copy()
    v_ref = vc.float().numpy().copy()
    for b in range(B):
        L = int(acc_len[b])
        oracle_compact(k_ref[:, b], v_ref[:, b], int(n_old[b]), acc_path[b, :L].tolist())
    kd, vd = kc.to(DEV), vc.to(DEV)
    api.compact(kd, vd, n_old.to(DEV), acc_len.to(DEV), acc_path.to(DEV))
    assert np.array_equal(kd.cpu().float().numpy(), k_ref)
    assert np.array_equal(vd.cpu().float().numpy(), v_ref)


@pytest.mark.parametrize("nq,nkv,T,ctx", [(40, 40, 49, 4100), (32, 8, 61, 1300), (32, 32, 1, 700)])
def test_attention_split_kv_long_context(nq, nkv, T, ctx):
    """Long-context tree/causal attention (split-KV with the log-sum-exp combine) equals the
    oracle, and equals the single-split result within bf16 output rounding."""
    g = torch.Generator().manual_seed(ctx)
    rng = np.random.default_rng(ctx)
    d, cap = 128, ctx + T + 8
    kc = _rand((1, nkv, cap, d), g, torch.bfloat16)
    vc = _rand((1, nkv, cap, d), g, torch.bfloat16)
    q = _rand((T, nq, d), g, torch.bfloat16)
    parent = [-1] + [int(rng.integers(0, i)) for i in range(1, T)]
    m = np.zeros((T, T), dtype=bool)
    for i in range(T):
        a = i
        while a >= 0:
            m[i, a] = True
            a = parent[a]
    mask = _mask_words(m).to(DEV)
    ctx_len = torch.tensor([ctx], dtype=torch.int32, device=DEV)
    row_seq = torch.zeros(T, dtype=torch.int32, device=DEV)
    row_slot = (ctx + torch.arange(T, dtype=torch.int32)).to(DEV)
    args = (q.to(DEV), kc.to(DEV), vc.to(DEV), row_seq, row_slot, ctx_len, T, 1, T, mask)
    split = api.attention(*args).cpu().double().numpy()
    vis = np.zeros((T, ctx + T), dtype=bool)
    vis[:, :ctx] = True
    vis[:, ctx:] = m
    want = oracle_attention(q.double().numpy(), kc[0, :, :ctx + T].double().numpy(),
                            vc[0, :, :ctx + T].double().numpy(), vis)
    assert np.max(np.abs(split - want)) < 2e-2


def _random_tree(rng, T):
    parent = [-1] + [int(rng.integers(0, i)) for i in range(1, T)]
    m = np.zeros((T, T), dtype=bool)
    for i in range(T):
        a = i
        while a >= 0:
            m[i, a] = True
            a = parent[a]
    return parent, m


@pytest.mark.parametrize("nq,nkv,d,T,ctx", [(32, 8, 128, 61, 1300), (32, 32, 128, 61, 700), (8, 2, 32, 17, 40),
                                            (5, 5, 64, 13, 9), (40, 40, 128, 49, 4100)])
def test_tree_row_equals_causal_row_bitwise(nq, nkv, d, T, ctx):
    """A tree row and plain causal decoding of the same token over the compacted cache (the
    context, then the row's root-to-node path in consecutive slots) give bit-identical
    attention outputs: the row's keys are summed in a decomposition fixed by its position
    alone, whatever the other rows of the launch are. The capacity is the same for both
    calls, as in an engine, where it fixes the key splits."""
    g = torch.Generator().manual_seed(ctx + T)
    rng = np.random.default_rng(ctx + T)
    cap = ctx + T + 40
    kc = _rand((1, nkv, cap, d), g, torch.bfloat16)
    vc = _rand((1, nkv, cap, d), g, torch.bfloat16)
    q = _rand((T, nq, d), g, torch.bfloat16)
    parent, m = _random_tree(rng, T)
    tree = api.attention(q.to(DEV), kc.to(DEV), vc.to(DEV), torch.zeros(T, dtype=torch.int32, device=DEV),
                         (ctx + torch.arange(T, dtype=torch.int32)).to(DEV),
                         torch.tensor([ctx], dtype=torch.int32, device=DEV), T, 1, T, _mask_words(m).to(DEV)).cpu()
    for i in sorted({0, T - 1, int(np.argmax(m.sum(1)))} | set(rng.integers(0, T, 4).tolist())):
        path = [j for j in range(T) if m[i, j]]            # root .. i, increasing depth
        kp, vp = kc.clone(), vc.clone()
        kp[0, :, ctx:ctx + len(path)] = kc[0, :, ctx + np.array(path)]
        vp[0, :, ctx:ctx + len(path)] = vc[0, :, ctx + np.array(path)]
        slot = ctx + len(path) - 1
        plain = api.attention(q[i:i + 1].to(DEV), kp.to(DEV), vp.to(DEV), torch.zeros(1, dtype=torch.int32, device=DEV),
                              torch.tensor([slot], dtype=torch.int32, device=DEV),
                              torch.zeros(1, dtype=torch.int32, device=DEV), 1, 0).cpu()
        assert torch.equal(plain[0], tree[i]), f"row {i} (depth {len(path) - 1})"


@pytest.mark.parametrize("N,K", [(4096, 4096), (1536, 1024), (520, 2056)])
def test_gemm_rows_do_not_depend_on_the_other_rows(N, K):
    """A token's projection is bit-identical in GEMMs of 1, 61, 300 and 1088 rows (one to
    five 256-row token tiles): the k-split points follow (N, K, SM count) only."""
    g = torch.Generator().manual_seed(N + K)
    X = _rand((1088, K), g, torch.bfloat16).to(DEV)
    W = _rand((N, K), g, torch.bfloat16, 0.05).to(DEV)
    full = api.gemm(W, X)
    for M in (1, 61, 300):
        for r0 in (0, 777):
            sub = api.gemm(W, X[r0:r0 + M].contiguous())
            assert torch.equal(sub, full[r0:r0 + M]), (M, r0)
    # the paired gate/up layout with the SwiGLU epilogue: the same rows, the same bits
    Wgu = _rand((2 * N, K), g, torch.bfloat16, 0.05).to(DEV) if N % 64 == 0 else None
    if Wgu is not None:
        big = api.gemm(Wgu, X, epi=4)
        for M in (1, 64):
            assert torch.equal(api.gemm(Wgu, X[5:5 + M].contiguous(), epi=4), big[5:5 + M])


@pytest.mark.parametrize("M,F,K", [(61, 11008 // 4, 1024), (10, 832, 320), (1, 640, 256), (130, 704, 264)])
def test_gemm_bf16_swiglu_epilogue(M, F, K):
    """Gate/up projection with SwiGLU in the epilogue: bf16(silu(X Wg^T) * (X Wu^T))."""
    g = torch.Generator().manual_seed(F + M)
    X = _rand((M, K), g, torch.bfloat16)
    W = _rand((2 * F, K), g, torch.bfloat16, 0.05)
    out = torch.zeros(M, F, dtype=torch.bfloat16, device=DEV)
    api.gemm(W.to(DEV), X.to(DEV), epi=4, out=out)
    x, w = X.double().numpy(), W.double().numpy()
    gate, up = x @ w[:F].T, x @ w[F:].T
    want = gate / (1 + np.exp(-gate)) * up
    mag = (np.abs(x) @ np.abs(w[:F]).T) * (np.abs(x) @ np.abs(w[F:]).T)
    got = out.cpu().double().numpy()
    assert np.all(np.abs(got - want) <= np.abs(want) * 2.0 ** -8 + 2e-3 * mag + 1e-6)
