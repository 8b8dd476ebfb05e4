"""The tcgen05 attention bodies (head dim 128, EAGLE_ATTN_TC=1), which the library selects
once per process: the kernel-level attention parity tests (against the oracle, and tree row =
causal row bit for bit), full-size greedy losslessness, and paged = contiguous at the 8B shape
(the paged cache's per-block TMA boxes) run again in a child process with the switch on."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_tcgen05_attention_bodies_pass_the_attention_parity_tests():
    env = dict(os.environ, EAGLE_ATTN_TC="1")
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_gpu_ops.py"), "-m", "gpu",
                        "-x", "-q", "-k", "attention or tree_row"], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert " passed" in r.stdout and "failed" not in r.stdout


def test_tcgen05_attention_bodies_keep_greedy_speculation_lossless():
    env = dict(os.environ, EAGLE_ATTN_TC="1")
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_gpu_fullshape.py"), "-m",
                        "gpu", "-x", "-q", "-k", "spec_equals_plain and 7b"], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert " passed" in r.stdout


def test_tcgen05_attention_bodies_paged_equals_contiguous():
    env = dict(os.environ, EAGLE_ATTN_TC="1")
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_gpu_paged.py"), "-m",
                        "gpu", "-x", "-q", "-k", "paged_equals_contiguous_full_size"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert " passed" in r.stdout
