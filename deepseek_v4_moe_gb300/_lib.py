"""ctypes binding of libmoe_ffn.so (the C ABI in include/moe_ffn.h): argument marshalling only.

Every step of the block runs in the library's CUDA kernels.  There is no Python or CPU fallback: if
the library cannot be built or loaded, ``load()`` raises.
"""
from __future__ import annotations

import ctypes
import os
import re

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_ffn.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "moe_ffn.h")

c_i32, c_f32, c_vp = ctypes.c_int32, ctypes.c_float, ctypes.c_void_p


class MoeFfnConfig(ctypes.Structure):
    _fields_ = [("hidden", c_i32), ("hc", c_i32), ("experts", c_i32), ("top_k", c_i32), ("inter", c_i32),
                ("shared_inter", c_i32), ("vocab", c_i32), ("n_layers", c_i32), ("hash_layer_count", c_i32),
                ("max_rows", c_i32), ("sinkhorn_iters", c_i32), ("rms_eps", c_f32)]


WEIGHT_FIELDS = ["hc_fn", "hc_base", "hc_scale", "ffn_norm", "gate", "exp_probs_b", "tid2eid", "gate_exps",
                 "up_exps", "down_exps", "gate_sh", "up_sh", "down_sh"]


class MoeFfnLayerWeights(ctypes.Structure):
    _fields_ = [(n, c_vp) for n in WEIGHT_FIELDS]


class MoeFfnHcWeights(ctypes.Structure):
    _fields_ = [("hc_fn", c_vp), ("hc_base", c_vp), ("hc_scale", c_vp), ("norm", c_vp)]


SUBLAYER_ATTN, SUBLAYER_FFN = 0, 1

MXFP8_FIELDS = ["gate_exps", "gate_exps_scale", "up_exps", "up_exps_scale", "down_exps", "down_exps_scale",
                "gate_sh", "gate_sh_scale", "up_sh", "up_sh_scale", "down_sh", "down_sh_scale"]


class MoeFfnMxfp8Experts(ctypes.Structure):
    _fields_ = [(n, c_vp) for n in MXFP8_FIELDS]

# return codes and device status bits (include/moe_ffn.h)
OK, ERR_NULL_PTR, ERR_BAD_CONFIG, ERR_LAYER_RANGE, ERR_ROWS_ZERO, ERR_ROWS_RANGE = 0, -1, -2, -3, -4, -5
ERR_NO_ROUTING_SOURCE, ERR_ALIAS, ERR_CUDA, ERR_NO_MEMORY, ERR_UNSUPPORTED, ERR_ALIGNMENT, ERR_NO_WEIGHTS = (
    -6, -7, -8, -9, -10, -11, -12)
DEV_TOKEN_RANGE, DEV_ROUTE_RANGE, DEV_NONFINITE, DEV_TIMEOUT = 0x1, 0x2, 0x4, 0x8

_lib = None


def declared_functions() -> list[str]:
    """Names of the functions include/moe_ffn.h declares."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:int|void|const char \*)\s*(moe_ffn_\w+)\s*\(", text, re.M)))


def load(build: bool = True):
    """Loads the library, building it first when it is missing or older than its sources."""
    global _lib
    if _lib is not None:
        return _lib
    if build:
        from . import build as _build
        try:
            _build.build()
        except RuntimeError:
            if not os.path.exists(LIB_PATH):
                raise
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with python -m deepseek_v4_moe_gb300.build")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32 = c_vp, c_i32
    lib.moe_ffn_init.argtypes = [ctypes.POINTER(MoeFfnConfig), ctypes.POINTER(MoeFfnLayerWeights),
                                 ctypes.POINTER(vp)]
    lib.moe_ffn_init.restype = ctypes.c_int
    lib.moe_ffn_forward.argtypes = [vp, vp, vp, i32, i32, vp, vp]
    lib.moe_ffn_forward.restype = ctypes.c_int
    lib.moe_ffn_forward_layers.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp]
    lib.moe_ffn_forward_layers.restype = ctypes.c_int
    lib.moe_ffn_forward_host.argtypes = [vp, vp, vp, i32, i32, vp, vp]
    lib.moe_ffn_forward_host.restype = ctypes.c_int
    lib.moe_ffn_status.argtypes = [vp]
    lib.moe_ffn_status.restype = ctypes.c_int
    lib.moe_ffn_debug_copy.argtypes = [vp, i32, vp, ctypes.c_size_t]
    lib.moe_ffn_debug_copy.restype = ctypes.c_int
    lib.moe_ffn_set_stage_timing.argtypes = [vp, i32]
    lib.moe_ffn_set_stage_timing.restype = ctypes.c_int
    lib.moe_ffn_stage_times.argtypes = [vp, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_char_p), i32]
    lib.moe_ffn_stage_times.restype = ctypes.c_int
    lib.moe_ffn_hc_split_noalloc.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, c_f32, vp, vp, vp, vp]
    lib.moe_ffn_hc_split_noalloc.restype = ctypes.c_int
    lib.moe_ffn_set_mxfp8_experts.argtypes = [vp, i32, ctypes.POINTER(MoeFfnMxfp8Experts)]
    lib.moe_ffn_set_mxfp8_experts.restype = ctypes.c_int
    lib.moe_ffn_set_attn_hc.argtypes = [vp, i32, ctypes.POINTER(MoeFfnHcWeights)]
    lib.moe_ffn_set_attn_hc.restype = ctypes.c_int
    lib.moe_ffn_hc_pre.argtypes = [vp, i32, i32, vp, i32, vp, vp, vp, vp, vp]
    lib.moe_ffn_hc_pre.restype = ctypes.c_int
    lib.moe_ffn_hc_post.argtypes = [vp, vp, vp, vp, vp, i32, vp, vp]
    lib.moe_ffn_hc_post.restype = ctypes.c_int
    lib.moe_ffn_set_fault_injection.argtypes = [vp, i32, ctypes.c_uint32]
    lib.moe_ffn_set_fault_injection.restype = ctypes.c_int
    lib.moe_ffn_last_error.argtypes = [vp]
    lib.moe_ffn_last_error.restype = ctypes.c_char_p
    lib.moe_ffn_destroy.argtypes = [vp]
    lib.moe_ffn_destroy.restype = None
    _lib = lib
    return lib
