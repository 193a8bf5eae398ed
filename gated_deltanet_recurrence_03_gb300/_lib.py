"""ctypes declarations of libgdn.so (the C ABI of include/gdn.h).

Loading fails loudly when the library has not been built: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgdn.so")

GDN_OK, GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED, GDN_ERR_CUDA, GDN_ERR_TIMEOUT, GDN_ERR_WORKSPACE = range(6)
GDN_F32, GDN_BF16 = 0, 1
GDN_NORMALIZE_QK = 0x1
GDN_RAW_GATES = 0x2
GDN_OUTPUT_GATE = 0x4

EXPORTED = ("gdn_opts_init", "gdn_chunk_fwd", "gdn_chunk_fwd_workspace_size", "gdn_recurrent_step",
            "gdn_check_device_status", "gdn_status_string", "gdn_last_error", "gdn_version",
            "gdn_chunk_fwd_noalloc", "gdn_causal_conv1d_fwd", "gdn_causal_conv1d_step",
            "gdn_recurrent_bwd", "gdn_recurrent_bwd_workspace_size", "gdn_causal_conv1d_fwd_qkv",
            "gdn_causal_conv1d_step_qkv", "gdn_output_gate_fwd", "gdn_output_gate_bwd",
            "gdn_output_gate_bwd_workspace_size", "gdn_causal_conv1d_bwd", "gdn_causal_conv1d_bwd_workspace_size")


class GdnOpts(ctypes.Structure):
    _fields_ = [
        ("dtype", ctypes.c_int),
        ("chunk", ctypes.c_int),
        ("scale", ctypes.c_float),
        ("flags", ctypes.c_uint),
        ("cu_seqlens", ctypes.c_void_p),
        ("num_seqs", ctypes.c_int),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
        ("stream", ctypes.c_void_p),
        ("events", ctypes.POINTER(ctypes.c_void_p)),
        ("num_events", ctypes.c_int),
        ("A_log", ctypes.c_void_p),
        ("dt_bias", ctypes.c_void_p),
        ("z", ctypes.c_void_p),
        ("norm_weight", ctypes.c_void_p),
        ("norm_eps", ctypes.c_float),
        ("grad_A_log", ctypes.c_void_p),
        ("grad_dt_bias", ctypes.c_void_p),
    ]


class GdnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"libgdn status {status}: {message}")
        self.status = status


_lib = None


def load(path: str = LIB_PATH):
    """Load libgdn.so and declare its entry points (cached)."""
    global _lib
    if _lib is not None and path == LIB_PATH:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"libgdn.so is not built ({path}); run __graft_entry__.build() "
                          "or python -m gated_deltanet_recurrence_03_gb300.build")
    lib = ctypes.CDLL(path)
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    opts_p = ctypes.POINTER(GdnOpts)
    lib.gdn_opts_init.argtypes = [opts_p]
    lib.gdn_opts_init.restype = None
    lib.gdn_chunk_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, opts_p]
    lib.gdn_chunk_fwd.restype = i
    lib.gdn_chunk_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, opts_p]
    lib.gdn_chunk_fwd_noalloc.restype = i
    ll = ctypes.c_longlong
    lib.gdn_causal_conv1d_fwd.argtypes = [vp, ll, vp, vp, vp, vp, i, i, i, i, opts_p]
    lib.gdn_causal_conv1d_fwd.restype = i
    lib.gdn_causal_conv1d_step.argtypes = [vp, ll, vp, vp, vp, i, i, i, opts_p]
    lib.gdn_causal_conv1d_step.restype = i
    lib.gdn_causal_conv1d_fwd_qkv.argtypes = [vp, ll, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, opts_p]
    lib.gdn_causal_conv1d_fwd_qkv.restype = i
    lib.gdn_causal_conv1d_step_qkv.argtypes = [vp, ll, vp, vp, vp, vp, vp, i, i, i, i, i, opts_p]
    lib.gdn_causal_conv1d_step_qkv.restype = i
    lib.gdn_recurrent_bwd.argtypes = [vp] * 14 + [i, i, i, i, i, i, opts_p]
    lib.gdn_recurrent_bwd.restype = i
    lib.gdn_output_gate_fwd.argtypes = [vp, vp, vp, vp, ll, i, opts_p]
    lib.gdn_output_gate_fwd.restype = i
    lib.gdn_output_gate_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, ll, i, opts_p]
    lib.gdn_output_gate_bwd.restype = i
    lib.gdn_output_gate_bwd_workspace_size.argtypes = [ll, i, opts_p]
    lib.gdn_output_gate_bwd_workspace_size.restype = ctypes.c_size_t
    lib.gdn_causal_conv1d_bwd.argtypes = [vp, ll, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, opts_p]
    lib.gdn_causal_conv1d_bwd.restype = i
    lib.gdn_causal_conv1d_bwd_workspace_size.argtypes = [i, i, i, i, opts_p]
    lib.gdn_causal_conv1d_bwd_workspace_size.restype = ctypes.c_size_t
    lib.gdn_recurrent_bwd_workspace_size.argtypes = [i, i, i, i, i, i, opts_p]
    lib.gdn_recurrent_bwd_workspace_size.restype = ctypes.c_size_t
    lib.gdn_chunk_fwd_workspace_size.argtypes = [i, i, i, i, i, i, opts_p]
    lib.gdn_chunk_fwd_workspace_size.restype = ctypes.c_size_t
    lib.gdn_recurrent_step.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, opts_p]
    lib.gdn_recurrent_step.restype = i
    lib.gdn_check_device_status.argtypes = [vp]
    lib.gdn_check_device_status.restype = i
    lib.gdn_status_string.argtypes = [i]
    lib.gdn_status_string.restype = ctypes.c_char_p
    lib.gdn_last_error.argtypes = []
    lib.gdn_last_error.restype = ctypes.c_char_p
    lib.gdn_version.argtypes = []
    lib.gdn_version.restype = i
    if path == LIB_PATH:
        _lib = lib
    return lib


def check(lib, status: int) -> None:
    if status != GDN_OK:
        msg = lib.gdn_last_error().decode() or lib.gdn_status_string(status).decode()
        raise GdnError(status, msg)


def default_opts(lib) -> GdnOpts:
    o = GdnOpts()
    lib.gdn_opts_init(ctypes.byref(o))
    return o
