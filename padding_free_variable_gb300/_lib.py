"""ctypes declarations of the C ABI in include/lstm_packed.h.

Argument marshalling only.  Loading fails loudly when the CUDA library has
not been built: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "liblstm_packed.so")

LSTM_OK = 0
LSTM_ERR_INVALID_ARG = 1
LSTM_ERR_UNSUPPORTED = 2
LSTM_ERR_CUDA = 3
LSTM_ERR_TIMEOUT = 4
LSTM_ERR_BOUNDS = 5
LSTM_F32 = 0
LSTM_BF16 = 1

# Every symbol the header declares, for the export check.
EXPORTED = (
    "lstm_plan_create", "lstm_plan_create_padded", "lstm_plan_destroy", "lstm_plan_info",
    "lstm_plan_tables", "lstm_plan_set_wait_limit", "lstm_workspace_bytes", "lstm_scratch_bytes",
    "lstm_pack", "lstm_unpack", "lstm_fwd", "lstm_bwd", "lstm_status_poll", "lstm_status_string",
    "lstm_debug_skip_arrival", "lstm_plan_dims", "lstm_plan_compute_host",
    "lstm_plan_set_ctas_per_direction", "lstm_plan_enable_timing", "lstm_plan_read_timing",
    "lstm_plan_launch_count", "lstm_debug_trace_steps", "lstm_bwd_noalloc",
    "lstm_plan_set_gemm_engine", "lstm_debug_input_projection", "lstm_plan_recurrent_config",
    "lstm_stepwise_scratch_bytes", "lstm_fwd_stepwise", "lstm_bwd_stepwise", "lstm_debug_cluster_variant",
    "lstm_plan_recurrent_groups", "lstm_debug_sequence_groups", "lstm_state_scratch_bytes", "lstm_fwd_state",
    "lstm_bwd_state", "lstm_plan_create_segments", "lstm_segments_host", "lstm_plan_create_window",
    "lstm_form_batches", "lstm_debug_wide_recurrence", "lstm_debug_wide_stages",
    "lstm_md_plan_create", "lstm_md_plan_compute_host", "lstm_md_plan_destroy", "lstm_md_plan_info",
    "lstm_md_plan_placement", "lstm_md_plan_step_cells", "lstm_md_plan_set_wait_limit", "lstm_md_status_poll",
    "lstm_md_plan_launch_count", "lstm_md_workspace_bytes", "lstm_md_scratch_bytes", "lstm_md_fwd", "lstm_md_bwd",
    "lstm_md_plan_enable_timing", "lstm_md_plan_read_timing", "lstm_md_debug_skip_arrival",
)

KERNEL_KINDS = ("pack", "unpack", "input_gemm", "rec_fwd", "rec_bwd", "gemm_dx", "gemm_dw", "gemm_dr", "convert")
MD_KINDS = ("md_input", "md_fwd", "md_bwd", "md_grads")


class LayerShape(ctypes.Structure):
    _fields_ = [("input_size", ctypes.c_int32), ("hidden_size", ctypes.c_int32),
                ("num_directions", ctypes.c_int32), ("dtype", ctypes.c_int32)]


class LayerParams(ctypes.Structure):
    _fields_ = [("W", ctypes.c_void_p), ("R", ctypes.c_void_p), ("b", ctypes.c_void_p),
                ("peep", ctypes.c_void_p)]


class LayerGrads(ctypes.Structure):
    _fields_ = [("dW", ctypes.c_void_p), ("dR", ctypes.c_void_p), ("db", ctypes.c_void_p),
                ("dpeep", ctypes.c_void_p)]


class State(ctypes.Structure):
    _fields_ = [("h0", ctypes.c_void_p), ("c0", ctypes.c_void_p)]


class StateGrads(ctypes.Structure):
    _fields_ = [("dh_n", ctypes.c_void_p), ("dc_n", ctypes.c_void_p), ("dh0", ctypes.c_void_p),
                ("dc0", ctypes.c_void_p)]


class MdShape(ctypes.Structure):
    _fields_ = [("input_size", ctypes.c_int32), ("hidden_size", ctypes.c_int32),
                ("num_directions", ctypes.c_int32)]


class MdParams(ctypes.Structure):
    _fields_ = [("W", ctypes.c_void_p), ("U1", ctypes.c_void_p), ("U2", ctypes.c_void_p), ("b", ctypes.c_void_p),
                ("peep", ctypes.c_void_p)]


class MdGrads(ctypes.Structure):
    _fields_ = [("W", ctypes.c_void_p), ("U1", ctypes.c_void_p), ("U2", ctypes.c_void_p), ("b", ctypes.c_void_p),
                ("peep", ctypes.c_void_p)]


class LSTMError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {status_string(code)} (status {code})")


_lib = None


def _declare(lib):
    vp, i32, i64, u64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_size_t
    pi32 = ctypes.POINTER(ctypes.c_int32)
    ppi32 = ctypes.POINTER(pi32)
    c = ctypes.c_int
    sig = {
        "lstm_plan_create": (c, [pi32, i32, ctypes.POINTER(vp)]),
        "lstm_plan_create_padded": (c, [pi32, i32, ctypes.POINTER(vp)]),
        "lstm_plan_destroy": (c, [vp]),
        "lstm_plan_info": (c, [vp, ctypes.POINTER(i64), pi32, pi32, ctypes.POINTER(i64)]),
        "lstm_plan_tables": (c, [vp, ppi32, ppi32, ppi32, ppi32]),
        "lstm_plan_set_wait_limit": (c, [vp, u64]),
        "lstm_workspace_bytes": (sz, [vp, ctypes.POINTER(LayerShape)]),
        "lstm_scratch_bytes": (sz, [vp, ctypes.POINTER(LayerShape)]),
        "lstm_pack": (c, [vp, vp, i32, i32, vp, vp]),
        "lstm_unpack": (c, [vp, vp, i32, i32, vp, vp]),
        "lstm_fwd": (c, [vp, ctypes.POINTER(LayerShape), ctypes.POINTER(LayerParams), vp, vp, vp, vp, vp,
                         vp, vp]),
        "lstm_bwd": (c, [vp, ctypes.POINTER(LayerShape), ctypes.POINTER(LayerParams), vp, vp, vp, vp, vp,
                         ctypes.POINTER(LayerGrads), vp, vp]),
        "lstm_status_poll": (c, [vp, vp]),
        "lstm_status_string": (ctypes.c_char_p, [c]),
        "lstm_debug_skip_arrival": (c, [vp, i32]),
        "lstm_debug_cluster_variant": (c, [vp, i32]),
        "lstm_plan_set_ctas_per_direction": (c, [vp, i32]),
        "lstm_plan_enable_timing": (c, [vp, i32]),
        "lstm_plan_read_timing": (c, [vp, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(i64)]),
        "lstm_plan_launch_count": (i64, [vp]),
        "lstm_plan_recurrent_config": (c, [vp, i32, pi32, pi32, pi32, pi32]),
        "lstm_plan_recurrent_groups": (c, [vp, i32, pi32, pi32]),
        "lstm_state_scratch_bytes": (sz, [vp, ctypes.POINTER(LayerShape)]),
        "lstm_plan_create_segments": (c, [pi32, i32, i32, i32, ctypes.POINTER(vp)]),
        "lstm_segments_host": (c, [pi32, i32, i32, i32, pi32, pi32, pi32, pi32, i32]),
        "lstm_plan_create_window": (c, [pi32, i32, i32, i32, ctypes.POINTER(vp)]),
        "lstm_form_batches": (c, [pi32, i32, i64, i32, pi32, pi32]),
        "lstm_fwd_state": (c, [vp, ctypes.POINTER(LayerShape), ctypes.POINTER(LayerParams), ctypes.POINTER(State),
                               vp, vp, vp, vp, vp, vp, vp, vp]),
        "lstm_bwd_state": (c, [vp, ctypes.POINTER(LayerShape), ctypes.POINTER(LayerParams), ctypes.POINTER(State),
                               vp, vp, vp, vp, vp, ctypes.POINTER(LayerGrads), ctypes.POINTER(StateGrads), vp, vp,
                               vp]),
        "lstm_debug_sequence_groups": (c, [vp, i32]),
        "lstm_debug_wide_recurrence": (c, [vp, i32]),
        "lstm_debug_wide_stages": (c, [vp, i32, pi32, pi32]),
        "lstm_md_plan_create": (c, [pi32, pi32, i32, i32, i32, i32, ctypes.POINTER(vp)]),
        "lstm_md_plan_compute_host": (c, [pi32, pi32, i32, i32, i32, i32, pi32, pi32, pi32,
                                          ctypes.POINTER(ctypes.c_int64), pi32, pi32, pi32, pi32, pi32]),
        "lstm_md_plan_destroy": (None, [vp]),
        "lstm_md_plan_info": (c, [vp, ctypes.POINTER(ctypes.c_int64), pi32, pi32, pi32, pi32]),
        "lstm_md_plan_placement": (c, [vp, pi32, pi32]),
        "lstm_md_plan_step_cells": (c, [vp, ctypes.POINTER(ctypes.c_int64)]),
        "lstm_md_plan_set_wait_limit": (c, [vp, u64]),
        "lstm_md_status_poll": (c, [vp, vp]),
        "lstm_md_plan_launch_count": (i64, [vp]),
        "lstm_md_plan_enable_timing": (c, [vp, i32]),
        "lstm_md_debug_skip_arrival": (c, [vp, i32]),
        "lstm_md_plan_read_timing": (c, [vp, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(i64)]),
        "lstm_md_workspace_bytes": (sz, [vp, ctypes.POINTER(MdShape)]),
        "lstm_md_scratch_bytes": (sz, [vp, ctypes.POINTER(MdShape)]),
        "lstm_md_fwd": (c, [vp, ctypes.POINTER(MdShape), ctypes.POINTER(MdParams), vp, vp, vp, vp]),
        "lstm_md_bwd": (c, [vp, ctypes.POINTER(MdShape), ctypes.POINTER(MdParams), vp, vp, vp, vp,
                            ctypes.POINTER(MdGrads), vp, vp]),
        "lstm_stepwise_scratch_bytes": (ctypes.c_size_t, [vp, ctypes.POINTER(LayerShape)]),
        "lstm_fwd_stepwise": (c, [vp, ctypes.POINTER(LayerShape), ctypes.POINTER(LayerParams), vp, vp, vp, vp, vp,
                                  vp, vp, vp]),
        "lstm_bwd_stepwise": (c, [vp, ctypes.POINTER(LayerShape), ctypes.POINTER(LayerParams), vp, vp, vp, vp, vp,
                                  ctypes.POINTER(LayerGrads), vp, vp]),
        "lstm_debug_trace_steps": (c, [vp, vp, i32]),
        "lstm_plan_set_gemm_engine": (c, [vp, i32]),
        "lstm_debug_input_projection": (c, [vp, ctypes.POINTER(LayerShape), ctypes.POINTER(LayerParams), vp, vp,
                                            vp]),
        "lstm_bwd_noalloc": (c, [vp, ctypes.POINTER(LayerShape), ctypes.POINTER(LayerParams), vp, vp, vp, vp, vp,
                                 ctypes.POINTER(LayerGrads), vp]),
        "lstm_plan_dims": (c, [pi32, i32, i32, pi32, ctypes.POINTER(i64)]),
        "lstm_plan_compute_host": (c, [pi32, i32, i32, pi32, pi32, pi32, pi32, pi32, pi32, pi32]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args


def load():
    """The loaded library; raises if it was not built (no CPU fallback exists)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with padding_free_variable_gb300.build.build() "
                               "(the packed LSTM has no CPU path)")
        lib = ctypes.CDLL(LIB_PATH)
        _declare(lib)
        _lib = lib
    return _lib


def status_string(code: int) -> str:
    try:
        return load().lstm_status_string(int(code)).decode()
    except Exception:  # pragma: no cover - library missing
        return "unknown"


def check(code: int, what: str):
    if code != LSTM_OK:
        raise LSTMError(code, what)
