"""The batch-aware draft budget planner (host arithmetic in the library; no GPU needed):
against a brute-force argmax over the same model of cost, and its expected behaviour -- free
verification takes the whole tree, rising verify cost shrinks the tree as the batch grows."""
import numpy as np
import pytest

from eagle_speculative_decoding_cycle_gb300 import _lib as L
from eagle_speculative_decoding_cycle_gb300 import api


@pytest.fixture(scope="module", autouse=True)
def _built():
    from eagle_speculative_decoding_cycle_gb300 import build
    build.build()


def _interp(rows_pts, us, rows):
    if len(rows_pts) == 1:
        return us[0] * max(1.0, rows / rows_pts[0])
    if rows <= rows_pts[0]:
        return us[0]
    for i in range(1, len(rows_pts)):
        if rows <= rows_pts[i]:
            f = (rows - rows_pts[i - 1]) / (rows_pts[i] - rows_pts[i - 1])
            return us[i - 1] + f * (us[i] - us[i - 1])
    slope = (us[-1] - us[-2]) / (rows_pts[-1] - rows_pts[-2])
    return us[-1] + max(0.0, slope) * (rows - rows_pts[-1])


def _brute(cands, rows_pts, us, B):
    best = (-1.0, None, None)
    for k, draft, ex in cands:
        for m in range(1, len(ex) + 1):
            r = B * np.float32(ex[m - 1]) / (np.float32(draft) + _interp(rows_pts, [np.float32(u) for u in us], B * (m + 1)))
            if r > best[0] + 1e-12 * max(1.0, abs(best[0])):
                best = (r, k, m)
    return best


def _curve(m_max, alpha):
    """Expected tokens of the m best nodes for a drafter whose i-th best node is accepted
    with probability alpha^(log2(i)+1): concave and increasing."""
    v = [alpha ** (np.log2(i) + 1) for i in range(1, m_max + 1)]
    return list(1.0 + np.cumsum(v))


def test_plan_matches_brute_force():
    rng = np.random.default_rng(3)
    for trial in range(30):
        cands = [(k, float(rng.uniform(200, 1500)), _curve(int(rng.integers(5, 60)), float(rng.uniform(0.5, 0.9))))
                 for k in (4, 8, 10)]
        n = int(rng.integers(1, 5))
        rows = sorted(set(int(x) for x in rng.integers(1, 5000, n)))
        us = sorted(float(x) for x in rng.uniform(500, 20000, len(rows)))
        B = int(rng.choice([1, 2, 8, 32, 64]))
        k, m, rate = api.plan_budget(cands, rows, us, B)
        r, kb, mb = _brute(cands, rows, us, B)
        assert rate == pytest.approx(r, rel=1e-5)
        assert (k, m) == (kb, mb)


def test_free_verification_takes_the_whole_tree():
    cands = [(10, 800.0, _curve(60, 0.8))]
    k, m, _ = api.plan_budget(cands, [1, 100000], [4000.0, 4000.0], 1)
    assert (k, m) == (10, 60)


def test_budget_shrinks_as_the_batch_grows():
    cands = [(10, 800.0, _curve(60, 0.8))]
    rows, us = [1, 128, 4096], [4000.0, 4100.0, 60000.0]   # weight-bound, then compute-bound
    ms = [api.plan_budget(cands, rows, us, B)[1] for B in (1, 4, 16, 64)]
    assert ms[0] == 60
    assert all(a >= b for a, b in zip(ms, ms[1:])) and ms[-1] < ms[0]


def test_bad_arguments_rejected():
    cands = [(10, 800.0, _curve(10, 0.8))]
    with pytest.raises(L.EagleError):
        api.plan_budget(cands, [100, 50], [1.0, 2.0], 1)      # rows not increasing
    with pytest.raises(L.EagleError):
        api.plan_budget(cands, [100], [0.0], 1)               # non-positive time
    with pytest.raises(L.EagleError):
        api.plan_budget(cands, [100], [10.0], 0)              # batch < 1
