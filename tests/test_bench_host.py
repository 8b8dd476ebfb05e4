"""Host-side logic of bench.py (no GPU): the algorithmic byte counts behind `hbm_gbs` and
the verify-pass fraction, and the static trees behind `--tree`."""
import bench
from eagle_speculative_decoding_cycle_gb300 import synth


def test_verify_bytes_of_the_7b_workload():
    """Layer weights 12.95 GB + LM head 0.262 GB + 648 context tokens of KV (512 KiB each)
    + 61 tree rows of KV written: 13.58 GB per verify pass."""
    wl = synth.LLAMA2_7B
    b = bench.algorithmic_bytes(wl, 648)
    kv_tok = 2 * 32 * 32 * 128 * 2
    assert kv_tok == 512 * 1024
    layers = 32 * (3 * 4096 * 4096 + 4096 * 4096 + 3 * 4096 * 11008) * 2
    assert b["verify_weights"] == layers + 32000 * 4096 * 2
    assert b["verify"] == layers + 32000 * 4096 * 2 + (648 + 61) * kv_tok
    assert abs(b["verify"] / 1e9 - 13.58) < 0.01


def test_batch_reads_weights_once_and_kv_per_sequence():
    wl = synth.LLAMA31_8B_BS64
    one = bench.algorithmic_bytes(wl, 1100, 1)
    many = bench.algorithmic_bytes(wl, 1100, 64)
    kv_tok = 2 * 32 * 8 * 128 * 2
    assert many["verify_weights"] == one["verify_weights"]
    assert many["verify"] - one["verify"] == 63 * (1100 + wl.tree.m + 1) * kv_tok
    assert many["cycle"] == many["verify"] + many["drafter"]


def _check_static(tree: synth.TreeShape):
    k, D = tree.topk, tree.depth
    parent, rank = tree.static_parent, tree.static_rank
    assert len(parent) == len(rank) == tree.m
    depth = []
    for i, (p, r) in enumerate(zip(parent, rank)):
        assert 0 <= r < k
        assert -1 <= p < i                     # parents come first: the kept set is closed
        depth.append(1 if p < 0 else depth[p] + 1)
    assert max(depth) <= D
    # at most k expanded nodes per depth, and no two children of one parent share a rank
    for d in range(1, D):
        assert len({p for p, dd in zip(parent, depth) if dd == d + 1}) <= k
    assert len(set(zip(parent, rank))) == len(parent)


def test_static_chain_is_one_rank0_child_per_depth():
    t = bench.static_tree("static-chain", synth.LLAMA2_7B.tree)
    D = synth.LLAMA2_7B.tree.depth
    assert t.m == D
    assert t.static_parent == tuple(range(-1, D - 1))
    assert t.static_rank == (0,) * D
    _check_static(t)


def test_static_prior_tree_is_a_valid_budgeted_tree():
    base = synth.LLAMA2_7B.tree
    t = bench.static_tree("static-prior", base)
    assert t.m == base.m
    _check_static(t)
    # best-first by prior: the root's rank-0 child comes first
    assert t.static_parent[0] == -1 and t.static_rank[0] == 0


def test_gemm_traffic_ratio_follows_the_source_digest(monkeypatch):
    """roofline traffic is scaled from the committed capture only while the GEMM sources it
    was taken on are the built ones."""
    from eagle_speculative_decoding_cycle_gb300 import build
    r = bench.traffic_ratio()
    assert r is not None and 0.95 < r < 1.1
    monkeypatch.setattr(build, "gemm_digest", lambda: "0000000000000000")
    assert bench.traffic_ratio() is None
