"""CPU oracle of the EAGLE / EAGLE-2 / EAGLE-3 draft-and-verify cycle.

TEST INFRASTRUCTURE. A plain, slow, obviously-correct numpy restatement of what
the cycle computes, written from the pages' description and used only to check
the CUDA path: only tests, `__graft_entry__.smoke()` and the CPU-baseline leg of
`bench.py` may import it. The product path never imports or calls it, and it
shares no code with the CUDA library; the only shared module is the seeded input
generator (`eagle_speculative_decoding_cycle_gb300.synth`), which holds no
arithmetic of the method.

Modules: philox (counter-based draws), model (target + drafters, fp64 with the
model's rounding points), tree (EAGLE-2 policy), accept (acceptance and KV
compaction), cycle (prefill, cycle, plain decode, planted mode), speedup (the
tokens-per-step model).

Parity status: every function is pinned by a test against what the pages or
mathematics fix (tests/test_oracle_*.py). The drafter's wiring (which feature and
which token feed a drafter position, which target layers EAGLE-3 fuses, and the
substitution of the drafter's own output below the root) is pinned by constructed
weights that reduce the drafter to an identity on one input, so its candidates follow
from the target alone (tests/test_oracle_wiring.py).
"""
