"""ctypes binding of libmmdit.so: the C ABI's structs and entry points.

Argument marshalling only.  Loading fails loudly when the shared library is
missing: there is no other implementation behind these names.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, Structure, c_double, c_float, c_int, c_int64, c_longlong, c_size_t, c_void_p

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmmdit.so")

MMDIT_OK = 0
MMDIT_BF16, MMDIT_F32, MMDIT_I8W, MMDIT_F8W = 0, 1, 2, 3
MMDIT_OP_DOUBLE, MMDIT_OP_SINGLE, MMDIT_OP_ATTENTION = 1, 2, 3
MMDIT_EPI_BF16, MMDIT_EPI_BF16_GELU, MMDIT_EPI_F32, MMDIT_EPI_RESID = 0, 1, 2, 3
ERRORS = {-1: "ARG", -2: "SHAPE", -3: "ALIGN", -4: "WORKSPACE", -5: "CUDA", -6: "TIMEOUT", -7: "UNSUPPORTED"}


class Shape(Structure):
    _fields_ = [("B", c_int), ("L_txt", c_int), ("grid_h", c_int), ("grid_w", c_int), ("D", c_int), ("H", c_int),
                ("d_head", c_int), ("D_mlp", c_int), ("rope_axes", c_int * 3), ("rope_theta", c_double),
                ("eps_ln", c_float), ("eps_rms", c_float), ("w_dtype", c_int), ("C_lat", c_int), ("t_dim", c_int),
                ("mlp_act", c_int), ("ref_h", c_int), ("ref_w", c_int)]


MMDIT_EPI_SWIGLU = 4
MMDIT_MLP_GELU = 0
MMDIT_MLP_SWIGLU = 1


class Linear(Structure):
    _fields_ = [("w", c_void_p), ("b", c_void_p), ("scale", c_void_p)]


class DoubleW(Structure):
    _fields_ = [("mod", Linear * 2), ("qkv", Linear * 2), ("proj", Linear * 2), ("mlp_in", Linear * 2),
                ("mlp_out", Linear * 2), ("q_norm", c_void_p * 2), ("k_norm", c_void_p * 2)]


class SingleW(Structure):
    _fields_ = [("mod", Linear), ("lin1", Linear), ("lin2", Linear), ("q_norm", c_void_p), ("k_norm", c_void_p)]


class StepW(Structure):
    _fields_ = [("time1", Linear), ("time2", Linear), ("img_in", Linear), ("final_mod", Linear), ("final", Linear),
                ("doubles", POINTER(DoubleW)), ("n_double", c_int), ("singles", POINTER(SingleW)),
                ("n_single", c_int)]


class CondW(Structure):
    _fields_ = [("txt_in", Linear), ("guid1", Linear), ("guid2", Linear), ("vec1", Linear), ("vec2", Linear),
                ("C_txt", c_int), ("C_pool", c_int)]


MMDIT_SAMPLE_GRAPH = 1

# name -> (restype, argtypes)
SIGNATURES = {
    "mmdit_status_string": (ctypes.c_char_p, [c_int]),
    "mmdit_sync_status": (c_int, [c_void_p]),
    "mmdit_launch_count": (c_longlong, []),
    "mmdit_selftest_wait_timeout": (c_int, [ctypes.c_uint, c_void_p]),
    "mmdit_kernel_name": (ctypes.c_char_p, [c_int]),
    "mmdit_trace_begin": (c_int, [c_int]),
    "mmdit_trace_end": (c_int, [POINTER(c_int)]),
    "mmdit_trace_read": (c_int, [POINTER(c_int), POINTER(c_float), c_int, POINTER(c_int)]),
    "mmdit_workspace_size": (c_int, [POINTER(Shape), c_int, POINTER(c_size_t)]),
    "mmdit_step_workspace_size": (c_int, [POINTER(Shape), c_int, c_int, POINTER(c_size_t)]),
    "mmdit_rope2d_build": (c_int, [POINTER(Shape), c_void_p, c_void_p, c_void_p, c_void_p]),
    "rope2d_apply": (c_int, [POINTER(Shape), c_void_p, c_void_p, c_void_p, c_int, c_void_p]),
    "joint_attention_fwd": (c_int, [POINTER(Shape), c_void_p, c_int, POINTER(c_void_p), POINTER(c_void_p), c_void_p,
                                    c_void_p, c_void_p, c_int, c_void_p, c_size_t, c_void_p]),
    "joint_attention_fwd_noalloc": (c_int, [POINTER(Shape), c_void_p, c_int, POINTER(c_void_p), POINTER(c_void_p),
                                            c_void_p, c_void_p, c_void_p, c_int, c_void_p]),
    "mmdit_double_block_fwd": (c_int, [POINTER(Shape), POINTER(DoubleW), c_void_p, c_void_p, c_void_p, c_void_p,
                                       c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "mmdit_single_block_fwd": (c_int, [POINTER(Shape), POINTER(SingleW), c_void_p, c_void_p, c_void_p, c_void_p,
                                       c_void_p, c_void_p, c_size_t, c_void_p]),
    "mmdit_step_fwd": (c_int, [POINTER(Shape), POINTER(StepW), c_void_p, c_void_p, c_double, c_double, c_void_p,
                               c_void_p, c_size_t, c_void_p]),
    "mmdit_step_i2i_fwd": (c_int, [POINTER(Shape), POINTER(StepW), c_void_p, c_void_p, c_void_p, c_double, c_double,
                                   c_void_p, c_void_p, c_size_t, c_void_p]),
    "mmdit_sample_workspace_size": (c_int, [POINTER(Shape), c_int, c_int, c_int, c_int, POINTER(c_size_t)]),
    "mmdit_sample": (c_int, [POINTER(Shape), POINTER(StepW), POINTER(CondW), c_void_p, c_void_p, c_void_p, c_double,
                             POINTER(c_double), c_int, c_int, c_void_p, c_size_t, c_void_p]),
    "euler_step": (c_int, [c_void_p, c_void_p, c_int, c_double, c_double, c_int64, c_void_p]),
    "mmdit_quantize_w8": (c_int, [c_void_p, c_int, c_int, c_int, c_void_p, c_void_p, c_void_p]),
    "mmdit_linear_fwd": (c_int, [POINTER(Linear), c_int, c_int, c_int, c_void_p, c_void_p, c_int, c_void_p, c_void_p,
                                 c_size_t, c_void_p]),
    "mmdit_quantize_f8": (c_int, [c_void_p, c_int, c_longlong, c_int, c_longlong, c_void_p, c_void_p, c_void_p]),
    "mmdit_linear_f8_fwd": (c_int, [POINTER(Linear), c_int, c_int, c_int, c_void_p, c_void_p, c_void_p, c_int,
                                    c_void_p, c_void_p]),
    "mmdit_ln_modulate": (c_int, [c_void_p, c_int, c_int, c_int, c_void_p, c_void_p, c_int64, c_float, c_void_p,
                                  c_void_p]),
    "mmdit_ln_modulate_f8": (c_int, [c_void_p, c_int, c_int, c_int, c_void_p, c_void_p, c_int64, c_float, c_void_p,
                                     c_void_p, c_void_p, c_void_p]),
    "mmdit_gemv": (c_int, [POINTER(Linear), c_int, c_int, c_int, c_void_p, c_int, c_void_p, c_void_p]),
    "mmdit_heads_pack": (c_int, [c_void_p, c_int64, c_int, c_int, c_int, c_int, c_void_p, c_void_p]),
    "mmdit_heads_unpack": (c_int, [c_void_p, c_int64, c_int, c_int, c_void_p, c_int, c_void_p]),
    "mmdit_shift_mu": (c_double, [c_int]),
    "mmdit_sigma_schedule": (c_int, [c_int, c_double, POINTER(c_double)]),
    "mmdit_time_embed": (c_int, [POINTER(Shape), POINTER(Linear), POINTER(Linear), c_double, c_void_p, c_void_p,
                                 c_void_p]),
}

_lib = None


def load(path: str = LIB_PATH):
    """Loads libmmdit.so and declares every entry point; raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libmmdit.so is not built ({path}); run diffusion_transformer_image_mmdit_gb300.build")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class MMDiTError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} returned {status} ({ERRORS.get(status, '?')})")
        self.status = status


def call(name: str, *args) -> None:
    st = getattr(load(), name)(*args)
    if st != MMDIT_OK:
        raise MMDiTError(name, st)
