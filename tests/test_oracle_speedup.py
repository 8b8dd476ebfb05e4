"""Pins of the tokens-per-step / speedup model against the numbers the pages print."""
import pytest

from conftest import golden_lines
from oracle.speedup import expected_tokens, speedup


def test_printed_speedups():
    n = 0
    for line in golden_lines("speedup_model.txt"):
        kind, a, c, k, tok, sp = line.split()
        a, c, k, tok, sp = float(a), float(c), int(k), float(tok), float(sp)
        if kind == "best":
            best = max(range(1, 7), key=lambda kk: speedup(a, kk, c))
            assert best == k
        assert round(expected_tokens(a, k), 2) == tok
        assert round(speedup(a, k, c), 2) == sp
        n += 1
    assert n == 4


def test_closed_form_geometric_sum():
    for a in (0.5, 0.8, 0.95):
        for k in (4, 5, 6):
            assert expected_tokens(a, k) == pytest.approx((1 - a ** (k + 1)) / (1 - a), rel=1e-12)
    # planted-mode expectations used by the bench (E[tau] = sum_{i<=D} p^i)
    assert round(expected_tokens(0.5, 6), 2) == 1.98
    assert round(expected_tokens(0.8, 6), 2) == 3.95
    assert round(expected_tokens(0.95, 6), 2) == 6.03
    assert round(expected_tokens(0.8, 4), 2) == 3.36
