"""ctypes mirror of include/evs.h and the loader of the in-tree ``libevs.so``.

Argument marshalling only: every step of the verify path runs inside the library's CUDA
kernels. If the library is missing the import of the handle fails loudly; there is no
fallback of any kind.
"""
from __future__ import annotations

import ctypes as C
import os

MAX_LAYERS = 64
PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libevs.so")

EVS_OK, EVS_ERR_INVALID_ARG, EVS_ERR_CAPACITY, EVS_ERR_STATE, EVS_ERR_CUDA = range(5)
LAYER_FIR, LAYER_IIR, LAYER_ATTN = 0, 1, 2
DTYPE_F32, DTYPE_BF16 = 0, 1
MODE_GREEDY, MODE_SAMPLING = 0, 1
CAND_RECURSIVE, CAND_MAX_ACCEPT = 0, 1
FLAG_KV_OVERFLOW, FLAG_BAD_K, FLAG_EMPTY_RESIDUAL, FLAG_BAD_TOKEN, FLAG_TIMEOUT = 1, 2, 4, 8, 16
(BUF_LOGITS, BUF_FIR_STAGE, BUF_IIR_U, BUF_K_CACHE, BUF_V_CACHE, BUF_K_SIDE, BUF_V_SIDE,
 BUF_KV_LEN, BUF_FIR_TAIL, BUF_IIR_STATE, BUF_CAND_K, BUF_CAND_CORR) = range(12)

EXPORTED = (
    "evs_workspace_bytes", "evs_create", "evs_destroy", "evs_set_stream", "evs_reset",
    "evs_prefill", "evs_verify_block", "evs_slice_state", "evs_replay_state", "evs_decode_step", "evs_import_state",
    "evs_export_state", "evs_debug_buffer", "evs_device_flags", "evs_last_launch_count",
    "evs_status_str", "evs_profile_enable", "evs_profile_read", "evs_debug_projection",
    "evs_projection_noalloc", "evs_projection_noalloc_flags",
)
KERNEL_KINDS = ("embed", "norm", "gemm", "fir", "iir", "kv_write", "attn", "attn_combine", "accept",
                "slice", "advance")


class Config(C.Structure):
    _fields_ = [("d", C.c_int32), ("vocab", C.c_int32), ("n_layers", C.c_int32),
                ("layer_kind", C.c_int32 * MAX_LAYERS), ("layer_param", C.c_int32 * MAX_LAYERS),
                ("head_dim", C.c_int32), ("gamma", C.c_int32), ("batch", C.c_int32),
                ("n_cand", C.c_int32), ("t_max", C.c_int32), ("prefill_chunk", C.c_int32),
                ("dtype", C.c_int32), ("mode", C.c_int32), ("temperature", C.c_float),
                ("near_tie_tau", C.c_float), ("cand_rule", C.c_int32)]


class LayerWeights(C.Structure):
    _fields_ = [("w_in", C.c_void_p), ("w_out", C.c_void_p), ("fir_taps", C.c_void_p),
                ("iir_lambda", C.c_void_p), ("iir_b", C.c_void_p), ("iir_c", C.c_void_p),
                ("w_qkv", C.c_void_p), ("w_o", C.c_void_p)]


class Weights(C.Structure):
    _fields_ = [("embed", C.c_void_p), ("head", C.c_void_p),
                ("layer", LayerWeights * MAX_LAYERS)]


class StateView(C.Structure):
    _fields_ = [("kv_len", C.POINTER(C.c_int32)), ("t_stride", C.c_int32),
                ("k", C.c_void_p * MAX_LAYERS), ("v", C.c_void_p * MAX_LAYERS),
                ("fir_tail", C.c_void_p * MAX_LAYERS), ("iir_state", C.c_void_p * MAX_LAYERS)]


class BufferInfo(C.Structure):
    _fields_ = [("ptr", C.c_void_p), ("bytes", C.c_size_t)]


_lib = None


def load(path: str = LIB_PATH) -> C.CDLL:
    """Load libevs.so (built by ``lossless_speculative_verify_gb300.build.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with lossless_speculative_verify_gb300.build.build() "
            "(nvcc, sm_103a). There is no non-CUDA implementation of this library.")
    lib = C.CDLL(path)
    vp, i32 = C.c_void_p, C.c_int32
    lib.evs_workspace_bytes.restype = C.c_size_t
    lib.evs_workspace_bytes.argtypes = [C.POINTER(Config)]
    lib.evs_create.restype = C.c_int
    lib.evs_create.argtypes = [C.POINTER(Config), C.POINTER(Weights), vp, C.c_size_t, vp,
                               C.POINTER(vp)]
    lib.evs_destroy.restype = None
    lib.evs_destroy.argtypes = [vp]
    lib.evs_set_stream.restype = C.c_int
    lib.evs_set_stream.argtypes = [vp, vp]
    lib.evs_reset.restype = C.c_int
    lib.evs_reset.argtypes = [vp]
    lib.evs_prefill.restype = C.c_int
    lib.evs_prefill.argtypes = [vp, vp, i32]
    lib.evs_verify_block.restype = C.c_int
    lib.evs_verify_block.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.evs_slice_state.restype = C.c_int
    lib.evs_slice_state.argtypes = [vp, vp, vp]
    lib.evs_replay_state.restype = C.c_int
    lib.evs_replay_state.argtypes = [vp, vp, vp, vp, vp]
    lib.evs_decode_step.restype = C.c_int
    lib.evs_decode_step.argtypes = [vp, vp, vp, vp, vp]
    lib.evs_import_state.restype = C.c_int
    lib.evs_import_state.argtypes = [vp, C.POINTER(StateView)]
    lib.evs_export_state.restype = C.c_int
    lib.evs_export_state.argtypes = [vp, C.POINTER(StateView)]
    lib.evs_debug_buffer.restype = C.c_int
    lib.evs_debug_buffer.argtypes = [vp, i32, i32, C.POINTER(BufferInfo)]
    lib.evs_device_flags.restype = C.c_int
    lib.evs_device_flags.argtypes = [vp, C.POINTER(C.c_uint32), i32]
    lib.evs_last_launch_count.restype = i32
    lib.evs_last_launch_count.argtypes = [vp]
    lib.evs_profile_enable.restype = C.c_int
    lib.evs_profile_enable.argtypes = [vp, i32]
    lib.evs_profile_read.restype = C.c_int
    lib.evs_profile_read.argtypes = [vp, C.POINTER(i32), C.POINTER(C.c_float), i32]
    lib.evs_debug_projection.restype = C.c_int
    lib.evs_debug_projection.argtypes = [vp, vp, i32, vp, vp, i32, i32, i32, i32, i32]
    lib.evs_projection_noalloc.restype = C.c_int
    lib.evs_projection_noalloc.argtypes = [vp, i32, vp, vp, i32, i32, i32, i32, i32, vp]
    lib.evs_projection_noalloc_flags.restype = C.c_int
    lib.evs_projection_noalloc_flags.argtypes = [C.POINTER(C.c_uint32), i32, vp]
    lib.evs_status_str.restype = C.c_char_p
    lib.evs_status_str.argtypes = [C.c_int]
    _lib = lib
    return lib


class EvsError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = load().evs_status_str(status).decode()
        super().__init__(f"{where}: {msg} (status {status})")
        self.status = status


def check(status: int, where: str) -> None:
    if status != EVS_OK:
        raise EvsError(status, where)
