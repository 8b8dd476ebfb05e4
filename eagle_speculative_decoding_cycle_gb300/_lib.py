"""ctypes declarations of the C ABI in include/eagle.h and include/eagle_ops.h.

Loading fails loudly when the CUDA library has not been built: there is no CPU or
eager fallback for any step of the cycle.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libeagle.so")

EAGLE_OK, EAGLE_EINVAL, EAGLE_ECAPACITY, EAGLE_ECUDA, EAGLE_EDEVICE, EAGLE_ETIMEOUT, EAGLE_EUNSUPPORTED = \
    0, -1, -2, -3, -4, -5, -6
STATUS_NAMES = {0: "EAGLE_OK", -1: "EAGLE_EINVAL", -2: "EAGLE_ECAPACITY", -3: "EAGLE_ECUDA",
                -4: "EAGLE_EDEVICE", -5: "EAGLE_ETIMEOUT", -6: "EAGLE_EUNSUPPORTED"}
DTYPE_F32, DTYPE_BF16 = 0, 1
DUMP_STATE, DUMP_CAND, DUMP_NODES, DUMP_TREE, DUMP_ACCEPT, DUMP_VERIFY_HEAD, DUMP_VERIFY_LOGITS, DUMP_FEATURES, \
    DUMP_TTT = range(9)
DEBUG_LOGITS = 1

# eagle_cycle_stats: six int32 counters, then the device clock at the cycle's start and at the
# end of each of its five phases (uint64 ns)
STATS_BYTES = 6 * 4 + 6 * 8
PHASES = ("draft", "select", "verify", "accept_compact", "update")

# every symbol the headers declare (checked by the CPU test suite)
EXPORTED = [
    "eagle_workspace_bytes", "eagle_create", "eagle_prefill", "eagle_cycle", "eagle_decode_plain",
    "eagle_set_graph", "eagle_set_stop", "eagle_set_tree_budget", "eagle_cycle_kernel_launches", "eagle_status_sync", "eagle_dump_bytes", "eagle_debug_dump", "eagle_set_debug",
    "eagle_kv_view", "eagle_kv_table", "eagle_set_static_tree", "eagle_ttt_forward", "eagle_profile_begin", "eagle_profile_end", "eagle_profile_verify", "eagle_profile_phases", "eagle_last_error", "eagle_destroy",
    "eagle_op_gemm_scratch_bytes", "eagle_op_gemm", "eagle_op_gemm_noalloc", "eagle_op_gemm_noalloc_status",
    "eagle_op_lm_head_scratch_bytes", "eagle_op_lm_head",
    "eagle_op_attention_scratch_bytes", "eagle_op_attention", "eagle_plan_budget", "eagle_op_tree_scratch_bytes", "eagle_op_tree_build", "eagle_op_compact",
    "eagle_op_wait_probe",
]


class ModelCfg(C.Structure):
    _fields_ = [("n_layers", C.c_int), ("hidden", C.c_int), ("n_heads", C.c_int), ("n_kv_heads", C.c_int),
                ("head_dim", C.c_int), ("ffn", C.c_int), ("vocab", C.c_int), ("rope_theta", C.c_float),
                ("rms_eps", C.c_float), ("dtype", C.c_int)]


class DrafterCfg(C.Structure):
    _fields_ = [("kind", C.c_int), ("fuse_layers", C.c_int * 3)]


class TreeCfg(C.Structure):
    _fields_ = [("topk", C.c_int), ("depth", C.c_int), ("m", C.c_int), ("temperature", C.c_float),
                ("seed", C.c_uint64), ("planted_p", C.c_float), ("planted_conf", C.c_float)]


class Limits(C.Structure):
    _fields_ = [("max_batch", C.c_int), ("max_ctx", C.c_int), ("kv_block", C.c_int), ("prefill_chunk", C.c_int)]


class LayerWeights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("attn_norm", "wqkv", "wo", "mlp_norm", "wgu", "wd")]


class Weights(C.Structure):
    _fields_ = [("embed", C.c_void_p), ("lm_head", C.c_void_p), ("final_norm", C.c_void_p),
                ("layers", C.POINTER(LayerWeights)), ("fc", C.c_void_p), ("norm_g", C.c_void_p),
                ("norm_e", C.c_void_p), ("draft", LayerWeights)]


_lib: Optional[C.CDLL] = None

vp, i32, u32, u64, f32, sz = C.c_void_p, C.c_int, C.c_uint32, C.c_uint64, C.c_float, C.c_size_t


def _declare(lib: C.CDLL) -> None:
    P = C.POINTER
    sig = {
        "eagle_workspace_bytes": (sz, [P(ModelCfg), P(DrafterCfg), P(TreeCfg), P(Limits)]),
        "eagle_create": (i32, [P(ModelCfg), P(DrafterCfg), P(TreeCfg), P(Weights), P(Limits), vp, sz, vp, P(vp)]),
        "eagle_prefill": (i32, [vp, i32, vp, P(C.c_int32), vp, i32]),
        "eagle_cycle": (i32, [vp, vp, vp, vp]),
        "eagle_decode_plain": (i32, [vp, i32, vp, vp]),
        "eagle_set_graph": (i32, [vp, i32]),
        "eagle_set_stop": (i32, [vp, i32, vp]),
        "eagle_set_tree_budget": (i32, [vp, i32, i32]),
        "eagle_cycle_kernel_launches": (i32, [vp]),
        "eagle_status_sync": (i32, [vp]),
        "eagle_dump_bytes": (sz, [vp, i32]),
        "eagle_debug_dump": (i32, [vp, i32, vp, sz]),
        "eagle_set_debug": (i32, [vp, i32]),
        "eagle_kv_view": (i32, [vp, P(vp), P(vp), P(i32)]),
        "eagle_kv_table": (i32, [vp, P(vp), P(i32), P(i32), P(i32)]),
        "eagle_set_static_tree": (i32, [vp, i32, P(i32), P(i32)]),
        "eagle_plan_budget": (i32, [i32, P(i32), P(C.c_float), P(i32), P(C.c_float), i32, P(i32), P(C.c_float), i32,
                                  P(i32), P(i32), P(C.c_float)]),
        "eagle_ttt_forward": (i32, [vp, vp, i32, i32, vp]),
        "eagle_profile_begin": (i32, [vp, i32]),
        "eagle_profile_end": (i32, [vp, P(i32), P(C.c_double), P(C.c_double)]),
        "eagle_profile_verify": (i32, [vp, P(i32), P(C.c_double)]),
        "eagle_profile_phases": (i32, [vp, P(i32), P(C.c_double)]),
        "eagle_last_error": (C.c_char_p, [vp]),
        "eagle_destroy": (None, [vp]),
        "eagle_op_gemm_scratch_bytes": (sz, [i32, i32]),
        "eagle_op_gemm": (i32, [i32, vp, vp, i32, i32, vp, i32, i32, vp, i32, vp, sz]),
        "eagle_op_gemm_noalloc": (i32, [vp, vp, i32, i32, vp, i32, i32, vp, i32]),
        "eagle_op_gemm_noalloc_status": (i32, [vp]),
        "eagle_op_lm_head_scratch_bytes": (sz, [i32, i32, i32, i32]),
        "eagle_op_lm_head": (i32, [i32, vp, vp, i32, i32, vp, i32, i32, f32, i32, i32, vp, i32, vp, vp, vp, u32,
                                   u64, i32, vp, vp, vp, vp, sz]),
        "eagle_op_attention_scratch_bytes": (sz, [i32, i32, i32]),
        "eagle_op_attention": (i32, [i32, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, vp, vp, vp, i32, i32,
                                     vp, i32, f32, i32, vp, sz]),
        "eagle_op_tree_scratch_bytes": (sz, [i32, i32, i32, i32]),
        "eagle_op_tree_build": (i32, [vp, i32, i32, i32, i32] + [vp] * 15 + [sz]),
        "eagle_op_compact": (i32, [i32, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp, i32]),
        "eagle_op_wait_probe": (i32, [vp, i32, vp, vp, vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args


def lib() -> C.CDLL:
    """The loaded library. Raises when libeagle.so is missing (build it with build())."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"CUDA library not built: {LIB_PATH} is missing "
                               "(run eagle_speculative_decoding_cycle_gb300.build.build())")
        l = C.CDLL(LIB_PATH)
        _declare(l)
        _lib = l
    return _lib


class EagleError(RuntimeError):
    def __init__(self, code: int, msg: str = ""):
        super().__init__(f"{STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


def check(code: int, msg: str = "") -> None:
    if code != EAGLE_OK:
        raise EagleError(code, msg)
