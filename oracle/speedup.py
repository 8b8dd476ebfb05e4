"""Oracle of the speculative-decoding speedup model.

Expected committed tokens per verify pass for a chain of k drafts, each accepted
with probability alpha given that the earlier ones were: 1 + alpha + ... +
alpha^k; speedup = that count / (1 + k * c), c being the cost of one draft pass
relative to one target pass ("EAGLE: Feature-Level Drafting", section "The math
behind the speedup with small numbers"; "Quick summary").

In planted mode every depth of the on-reference path is planted independently
with probability p, so the accepted length is the run of planted depths from
the root and the expected tokens per cycle is the same sum with alpha = p and
k = D (natural acceptance adds a little on top).

Test infrastructure: only tests, the smoke check and the bench's CPU baseline
use this package.
"""


def expected_tokens(alpha: float, k: int) -> float:
    """1 + alpha + ... + alpha^k: expected committed tokens per verify pass of a k-draft chain."""
    return sum(alpha ** i for i in range(k + 1))


def speedup(alpha: float, k: int, draft_cost: float) -> float:
    """expected_tokens / (1 + k * draft_cost), draft_cost = one draft pass relative to one target pass."""
    return expected_tokens(alpha, k) / (1.0 + k * draft_cost)
