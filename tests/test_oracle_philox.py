"""Pins of the oracle's counter-based generator and rounding helper."""
import numpy as np
import pytest
import torch

from conftest import golden_lines
from oracle import philox
from oracle.model import bf16_round


def test_philox_known_answers():
    n = 0
    for line in golden_lines("philox4x32_10_kat.txt"):
        lhs, rhs = line.split(":")
        w = [int(x, 16) for x in lhs.split()]
        want = [int(x, 16) for x in rhs.split()]
        got = philox.philox4x32_10(np.array(w[:4], np.uint64), np.array(w[4:], np.uint64))
        assert [int(x) for x in got] == want
        n += 1
    assert n == 3


def test_uniform_open_interval_and_exact():
    x = np.array([0, 255, 256, 0xFFFFFFFF], dtype=np.uint64)
    u = philox.to_uniform(x)
    assert np.all(u > 0) and np.all(u < 1)
    assert np.all(u.astype(np.float32).astype(np.float64) == u)   # exact in fp32


def test_gumbel_row_is_vectorised_scalar_draw():
    g = philox.gumbel_row(7, philox.STREAM_GUMBEL, 3, 11, 5, 10)
    for v in range(10):
        ctr = np.array([v >> 2, 5, 11, (3 << 8) | philox.STREAM_GUMBEL], np.uint64)
        u = philox.to_uniform(philox.philox4x32_10(ctr, philox.key_of(7))[v & 3])
        assert g[v] == pytest.approx(-np.log(-np.log(u)), abs=0)


def test_gumbel_distribution_moments():
    g = philox.gumbel_row(1, philox.STREAM_GUMBEL, 0, 0, 0, 200000)
    # Gumbel(0,1): mean = Euler-Mascheroni constant, variance = pi^2 / 6
    assert abs(g.mean() - 0.5772156649) < 0.01
    assert abs(g.var() - np.pi ** 2 / 6) < 0.03


def test_bf16_round_matches_torch_cast():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000) * 10.0 ** rng.integers(-8, 8, 100000),
                        [0.0, -0.0, 1.0, 1.00390625, 1.0078125, 65504.0]])
    want = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(bf16_round(x), want)
