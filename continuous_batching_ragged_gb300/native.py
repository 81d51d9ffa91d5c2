"""ctypes declarations of the C ABI in include/cb.h and include/cb_synth.h.

Loading fails loudly when ``libcb.so`` has not been built: there is no other
implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libcb.so")

CB_OK, CB_ERR_INVALID, CB_ERR_BOUNDS, CB_ERR_NO_BLOCKS, CB_ERR_TIMEOUT, CB_ERR_CUDA, CB_ERR_UNSUPPORTED = range(7)
STATUS_NAMES = {0: "CB_OK", 1: "CB_ERR_INVALID", 2: "CB_ERR_BOUNDS", 3: "CB_ERR_NO_BLOCKS",
                4: "CB_ERR_TIMEOUT", 5: "CB_ERR_CUDA", 6: "CB_ERR_UNSUPPORTED"}
CB_DTYPE_F32, CB_DTYPE_BF16 = 0, 1
NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024      # CB_NOALLOC_SCRATCH_BYTES in cb.h

# Every entry point declared in the public headers.
EXPORTS = ("cb_append_kv", "cb_attention_workspace_size", "cb_ragged_attention",
           "cb_append_kv_dims", "cb_plan_step", "cb_ragged_attention_planned",
           "cb_ragged_attention_gqa", "cb_attention_workspace_size_gqa",
           "cb_plan_step_gqa", "cb_ragged_attention_planned_gqa",
           "cb_decode_attention_noalloc", "cb_padded_attention",
           "cb_scheduler_create", "cb_scheduler_destroy", "cb_add_request", "cb_build_batch",
           "cb_complete_step", "cb_scheduler_stats", "cb_check_device_errors", "cb_last_error",
           "cb_synth_tokens", "cb_synth_fill_cache", "cb_selftest_bounded_wait")


CB_ADMIT_RESERVE_LIFETIME = 0
CB_ADMIT_PROMPT_PREEMPT = 1
ADMISSION = {"reserve_lifetime": CB_ADMIT_RESERVE_LIFETIME, "prompt_preempt": CB_ADMIT_PROMPT_PREEMPT}


class cb_kv_cache(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("num_blocks", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("num_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("dtype", ctypes.c_int)]


class cb_sched_config(ctypes.Structure):
    _fields_ = [("token_budget", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_blocks", ctypes.c_int32), ("max_num_seqs", ctypes.c_int32),
                ("admission", ctypes.c_int32)]


_P32 = ctypes.POINTER(ctypes.c_int32)
_P64 = ctypes.POINTER(ctypes.c_int64)


class cb_batch(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("num_tokens", ctypes.c_int32),
                ("num_decode", ctypes.c_int32), ("max_blocks_per_seq", ctypes.c_int32),
                ("max_q_len", ctypes.c_int32), ("max_context_len", ctypes.c_int32),
                ("cu_seqlens_q", _P32), ("context_lens", _P32), ("block_tables", _P32),
                ("slot_mapping", _P64), ("request_ids", _P64), ("num_evicted", ctypes.c_int32),
                ("evicted_ids", _P64), ("num_preempted", ctypes.c_int32), ("preempted_ids", _P64)]


class cb_sched_stats(ctypes.Structure):
    _fields_ = [("step", ctypes.c_int64), ("num_waiting", ctypes.c_int32),
                ("num_running", ctypes.c_int32), ("free_blocks", ctypes.c_int32),
                ("reserved_blocks", ctypes.c_int32), ("num_finished", ctypes.c_int64),
                ("num_preempted", ctypes.c_int64), ("recomputed_tokens", ctypes.c_int64)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "`python -m continuous_batching_ragged_gb300.build`")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, u64, f32, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64,
                                  ctypes.c_float, ctypes.c_size_t)
    st = ctypes.c_int
    pcache = ctypes.POINTER(cb_kv_cache)
    sigs = {
        "cb_append_kv": (st, [vp, vp, vp, i32, pcache, vp]),
        "cb_attention_workspace_size": (sz, [pcache, i32, i32, i32]),
        "cb_ragged_attention": (st, [vp, pcache, vp, vp, vp, i32, i32, i32, i32, i32, f32, vp, vp, sz, vp]),
        "cb_append_kv_dims": (st, [vp, vp, vp, vp, i32, pcache, vp]),
        "cb_ragged_attention_gqa": (st, [vp, i32, pcache, vp, vp, vp, i32, i32, i32, i32, i32, f32, vp, vp, sz,
                                         vp]),
        "cb_attention_workspace_size_gqa": (sz, [pcache, i32, i32, i32, i32]),
        "cb_padded_attention": (st, [vp, pcache, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, vp, vp, sz, vp]),
        "cb_plan_step": (st, [pcache, vp, vp, vp, i32, i32, i32, i32, i32, vp, sz, vp]),
        "cb_ragged_attention_planned": (st, [vp, pcache, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, vp, vp,
                                             sz, vp]),
        "cb_plan_step_gqa": (st, [pcache, i32, vp, vp, vp, i32, i32, i32, i32, i32, vp, sz, vp]),
        "cb_ragged_attention_planned_gqa": (st, [vp, i32, pcache, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32,
                                                 vp, vp, sz, vp]),
        "cb_decode_attention_noalloc": (st, [vp, pcache, vp, vp, vp, i32, i32, i32, i32, f32, vp, vp]),
        "cb_scheduler_create": (st, [ctypes.POINTER(cb_sched_config), ctypes.POINTER(vp)]),
        "cb_scheduler_destroy": (None, [vp]),
        "cb_add_request": (st, [vp, i64, i64, i32, i32]),
        "cb_build_batch": (st, [vp, ctypes.POINTER(cb_batch)]),
        "cb_complete_step": (st, [vp]),
        "cb_scheduler_stats": (st, [vp, ctypes.POINTER(cb_sched_stats)]),
        "cb_check_device_errors": (st, [vp]),
        "cb_last_error": (ctypes.c_char_p, []),
        "cb_selftest_bounded_wait": (st, [i32, vp]),
        "cb_synth_tokens": (st, [vp, ctypes.c_int, u64, i32, i32, vp, vp, i32, i32, i32, vp]),
        "cb_synth_fill_cache": (st, [vp, ctypes.c_int, u64, i32, i32, vp, vp, vp, i32, i32, i32, i32,
                                     i32, i32, i32, vp]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


class CBError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = lib().cb_last_error().decode(errors="replace")
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}: {msg}")


def check(status: int, where: str) -> None:
    if status != CB_OK:
        raise CBError(status, where)
