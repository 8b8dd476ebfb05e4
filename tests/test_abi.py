"""CPU checks of the C ABI: the library builds/loads, exports every declared symbol,
and sizes its workspace (pure host logic, no GPU needed)."""
import ctypes as C
import os
import re

import pytest

from conftest import ROOT
from eagle_speculative_decoding_cycle_gb300 import _lib as L
from eagle_speculative_decoding_cycle_gb300 import api, synth


def _declared():
    names = []
    for h in ("eagle.h", "eagle_ops.h"):
        txt = open(os.path.join(ROOT, "include", h)).read()
        txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
        names += re.findall(r"\b(eagle_[a-z0-9_]+)\s*\(", txt)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from eagle_speculative_decoding_cycle_gb300 import build
    build.build()
    return L.lib()


def test_exports_every_declared_symbol(lib):
    declared = _declared()
    assert sorted(L.EXPORTED) == declared
    for n in declared:
        assert hasattr(lib, n), n


def _cfg(w, **kw):
    return api.configs(w, **kw)


@pytest.mark.parametrize("w", [synth.TINY, synth.LLAMA2_7B, synth.LLAMA31_8B_SAMPLE, synth.LLAMA_13B_LONG,
                               synth.SMALL_BF16, synth.SMALL_BF16_E3])
def test_workspace_sizes(lib, w):
    mc, dc, tc, lim = _cfg(w)
    nb = lib.eagle_workspace_bytes(C.byref(mc), C.byref(dc), C.byref(tc), C.byref(lim))
    m = w.model
    es = 4 if m.dtype == "f32" else 2
    kv = 2 * m.n_layers * lim.max_batch * m.n_kv_heads * lim.max_ctx * m.head_dim * es
    assert nb > kv and nb < kv * 3 + (4 << 30)


def test_workspace_rejects_bad_configs(lib):
    w = synth.TINY
    for mutate in (lambda mc, dc, tc, lim: setattr(tc, "topk", 0),
                   lambda mc, dc, tc, lim: setattr(tc, "topk", 17),
                   lambda mc, dc, tc, lim: setattr(tc, "m", 10 ** 6),
                   lambda mc, dc, tc, lim: setattr(tc, "depth", 9),
                   lambda mc, dc, tc, lim: setattr(mc, "n_kv_heads", 3),
                   lambda mc, dc, tc, lim: setattr(mc, "head_dim", 256),
                   lambda mc, dc, tc, lim: setattr(dc, "kind", 2),
                   lambda mc, dc, tc, lim: setattr(lim, "kv_block", 12),
                   lambda mc, dc, tc, lim: setattr(lim, "kv_block", 4),
                   lambda mc, dc, tc, lim: setattr(lim, "kv_block", 512),
                   lambda mc, dc, tc, lim: setattr(lim, "kv_block", -16),
                   lambda mc, dc, tc, lim: setattr(tc, "planted_conf", 1.0)):
        mc, dc, tc, lim = _cfg(w)
        mutate(mc, dc, tc, lim)
        assert lib.eagle_workspace_bytes(C.byref(mc), C.byref(dc), C.byref(tc), C.byref(lim)) == 0


def test_paged_kv_workspace(lib):
    """kv_block = 16 (the batch-64 configuration's paged cache) is accepted; the pool holds
    every sequence's worst case, so it costs at most one block per sequence more than the
    contiguous cache."""
    w = synth.LLAMA31_8B_BS64
    assert w.kv_block == 16
    mc, dc, tc, lim = _cfg(w)
    paged = lib.eagle_workspace_bytes(C.byref(mc), C.byref(dc), C.byref(tc), C.byref(lim))
    lim.kv_block = 0
    contiguous = lib.eagle_workspace_bytes(C.byref(mc), C.byref(dc), C.byref(tc), C.byref(lim))
    assert paged > 0 and contiguous > 0
    m = w.model
    block_bytes = 2 * m.n_layers * m.n_kv_heads * 16 * m.head_dim * 2
    assert contiguous <= paged <= contiguous + lim.max_batch * (block_bytes + 64) + (1 << 20)


def test_create_rejects_without_touching_gpu(lib):
    """Argument errors are caught on the host before any CUDA call."""
    mc, dc, tc, lim = _cfg(synth.TINY)
    h = C.c_void_p()
    w = L.Weights()
    rc = lib.eagle_create(C.byref(mc), C.byref(dc), C.byref(tc), C.byref(w), C.byref(lim), None, 0, None, C.byref(h))
    assert rc == L.EAGLE_EINVAL and not h.value
    tc.topk = 0
    rc = lib.eagle_create(C.byref(mc), C.byref(dc), C.byref(tc), C.byref(w), C.byref(lim), None, 0, None, C.byref(h))
    assert rc == L.EAGLE_EINVAL


def test_injected_create_fault_fails_on_the_host(lib, monkeypatch):
    """EAGLE_FAULT=create makes a create call that passed every argument check fail with
    EAGLE_ECUDA before its first CUDA call (placeholder pointers are never dereferenced)."""
    mc, dc, tc, lim = _cfg(synth.TINY)
    fake = C.c_void_p(256)
    layers = (L.LayerWeights * mc.n_layers)()
    for lw in layers:
        for name, _ in L.LayerWeights._fields_:
            setattr(lw, name, fake)
    w = L.Weights()
    for name in ("embed", "lm_head", "final_norm", "fc", "norm_g", "norm_e"):
        setattr(w, name, fake)
    w.layers = layers
    for name, _ in L.LayerWeights._fields_:
        setattr(w.draft, name, fake)
    need = lib.eagle_workspace_bytes(C.byref(mc), C.byref(dc), C.byref(tc), C.byref(lim))
    assert need > 0
    monkeypatch.setenv("EAGLE_FAULT", "create")
    h = C.c_void_p()
    rc = lib.eagle_create(C.byref(mc), C.byref(dc), C.byref(tc), C.byref(w), C.byref(lim), fake, need, None,
                          C.byref(h))
    assert rc == L.EAGLE_ECUDA and not h.value
    # a workspace one byte short is refused first, fault or not
    rc = lib.eagle_create(C.byref(mc), C.byref(dc), C.byref(tc), C.byref(w), C.byref(lim), fake, need - 1, None,
                          C.byref(h))
    assert rc == L.EAGLE_ECAPACITY and not h.value


def test_op_scratch_sizes(lib):
    assert lib.eagle_op_gemm_scratch_bytes(61, 12288) > 0
    assert lib.eagle_op_gemm_scratch_bytes(0, 10) == 0
    assert lib.eagle_op_lm_head_scratch_bytes(1, 32000, 61, 2) > 0
    assert lib.eagle_op_lm_head_scratch_bytes(1, 32000, 61, 17) == 0
    assert lib.eagle_op_tree_scratch_bytes(1, 10, 6, 60) > 0
    assert lib.eagle_op_tree_scratch_bytes(1, 10, 9, 60) == 0


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(L, "LIB_PATH", str(tmp_path / "nope.so"))
    monkeypatch.setattr(L, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        L.lib()


def test_cycle_stats_layout_matches_the_header(tmp_path):
    """The binding's view of eagle_cycle_stats (its size, and the offsets read_stats decodes)
    equals the C struct of include/eagle.h, compiled here with the host compiler."""
    import shutil
    import subprocess
    import torch
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no host C compiler")
    src = tmp_path / "stats.c"
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "eagle.h"\n'
                   'int main(void) { printf("%zu %zu %zu %zu\\n", sizeof(eagle_cycle_stats),'
                   ' offsetof(eagle_cycle_stats, committed), offsetof(eagle_cycle_stats, verify_rows),'
                   ' offsetof(eagle_cycle_stats, t_ns)); return 0; }\n')
    exe = tmp_path / "stats"
    subprocess.check_call([cc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)])
    size, committed, rows, t_ns = map(int, subprocess.check_output([str(exe)]).split())
    assert size == L.STATS_BYTES and (committed, rows, t_ns) == (12, 20, 24)
    # read_stats on a buffer with known fields
    raw = torch.zeros(L.STATS_BYTES, dtype=torch.uint8)
    raw[:24].view(torch.int32).copy_(torch.tensor([3, 2, 5, 7, 4, 15], dtype=torch.int32))
    raw[24:].view(torch.int64).copy_(torch.tensor([1000, 3000, 3500, 9500, 10000, 12000], dtype=torch.int64))
    st = api.read_stats(raw)
    assert (st["batch"], st["active"], st["accepted"], st["committed"], st["max_accepted"], st["verify_rows"]) == \
        (3, 2, 5, 7, 4, 15)
    assert st["phase_us"] == {"draft": 2.0, "select": 0.5, "verify": 6.0, "accept_compact": 0.5, "update": 2.0}
    assert st["cycle_us"] == 11.0


def test_attention_op_rejects_a_batch_capacity_below_one(lib):
    """The attention op's engine batch capacity (which fixes its key-split length and the
    caches' TMA extent) must be >= 1; the check runs on the host before any launch."""
    fake = C.c_void_p(256)   # never dereferenced: the argument check returns first
    rc = lib.eagle_op_attention(L.DTYPE_BF16, None, fake, fake, fake, fake, 4, 32, 8, 128, 64, 4, fake, fake, fake,
                                0, 0, None, 0, 0.0, 0, fake, 1 << 20)
    assert rc == L.EAGLE_EINVAL
