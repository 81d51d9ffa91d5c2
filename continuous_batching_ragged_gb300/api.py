"""Thin Python binding of the C ABI: argument marshalling only.

Functions carry the C names.  Tensors are torch tensors on the current CUDA
device (torch supplies device memory and streams, nothing else); every step
of the computation runs in the library's kernels.
"""
from __future__ import annotations

import ctypes
import dataclasses
from typing import Optional

import numpy as np
import torch

from . import native
from .native import check

_DTYPES = {torch.bfloat16: native.CB_DTYPE_BF16, torch.float32: native.CB_DTYPE_F32}


def _stream_handle(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


@dataclasses.dataclass
class KVCache:
    """One layer's paged cache: k, v are [num_blocks, H, block_size, A] tensors."""
    k: torch.Tensor
    v: torch.Tensor

    def __post_init__(self):
        if self.k.shape != self.v.shape or self.k.dim() != 4 or self.k.dtype != self.v.dtype:
            raise ValueError("k and v must be equal-shaped [num_blocks, H, B, A] tensors")
        if self.k.dtype not in _DTYPES:
            raise ValueError(f"unsupported cache dtype {self.k.dtype}")

    @classmethod
    def empty(cls, num_blocks: int, num_heads: int, block_size: int, head_dim: int,
              dtype=torch.bfloat16, device="cuda") -> "KVCache":
        shape = (num_blocks, num_heads, block_size, head_dim)
        return cls(torch.empty(shape, dtype=dtype, device=device),
                   torch.empty(shape, dtype=dtype, device=device))

    @property
    def num_blocks(self) -> int:
        return self.k.shape[0]

    @property
    def num_heads(self) -> int:
        return self.k.shape[1]

    @property
    def block_size(self) -> int:
        return self.k.shape[2]

    @property
    def head_dim(self) -> int:
        return self.k.shape[3]

    def c_struct(self) -> native.cb_kv_cache:
        return native.cb_kv_cache(_ptr(self.k), _ptr(self.v), self.num_blocks, self.block_size,
                                  self.num_heads, self.head_dim, _DTYPES[self.k.dtype])


def cb_append_kv(k_new: torch.Tensor, v_new: torch.Tensor, slot_mapping: torch.Tensor,
                 cache: KVCache, stream=None) -> None:
    if slot_mapping.dtype != torch.int64:
        raise ValueError("slot_mapping must be int64")
    c = cache.c_struct()
    check(native.lib().cb_append_kv(_ptr(k_new), _ptr(v_new), _ptr(slot_mapping), k_new.shape[0],
                                    ctypes.byref(c), _stream_handle(stream)), "cb_append_kv")


def cb_attention_workspace_size(cache: KVCache, num_seqs: int, num_tokens: int,
                                max_context_len: int) -> int:
    c = cache.c_struct()
    return int(native.lib().cb_attention_workspace_size(ctypes.byref(c), num_seqs, num_tokens,
                                                        max_context_len))


def cb_ragged_attention(q: torch.Tensor, cache: KVCache, cu_seqlens_q: torch.Tensor,
                        context_lens: torch.Tensor, block_tables: torch.Tensor, *,
                        max_q_len: int, max_context_len: int, scale: float, out: torch.Tensor,
                        workspace: Optional[torch.Tensor], stream=None) -> torch.Tensor:
    for name, t in (("cu_seqlens_q", cu_seqlens_q), ("context_lens", context_lens),
                    ("block_tables", block_tables)):
        if t.dtype != torch.int32:
            raise ValueError(f"{name} must be int32")
    if block_tables.dim() != 2:
        raise ValueError("block_tables must be [num_seqs, max_blocks_per_seq]")
    c = cache.c_struct()
    ws_ptr = _ptr(workspace) if workspace is not None and workspace.numel() else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    check(native.lib().cb_ragged_attention(
        _ptr(q), ctypes.byref(c), _ptr(cu_seqlens_q), _ptr(context_lens), _ptr(block_tables),
        context_lens.shape[0], q.shape[0], block_tables.shape[1], max_q_len, max_context_len,
        float(scale), _ptr(out), ws_ptr, ws_bytes, _stream_handle(stream)), "cb_ragged_attention")
    return out


def cb_padded_attention(q: torch.Tensor, cache: KVCache, cu_seqlens_q: torch.Tensor,
                        context_lens: torch.Tensor, block_tables: torch.Tensor, pad_lens: torch.Tensor, *,
                        max_q_len: int, max_context_len: int, scale: float, out: torch.Tensor,
                        workspace: Optional[torch.Tensor], stream=None) -> torch.Tensor:
    """cb_padded_attention: a left-padded batch; the first pad_lens[s] rows of
    sequence s are padding (masked keys, rows not written)."""
    for name, t in (("cu_seqlens_q", cu_seqlens_q), ("context_lens", context_lens),
                    ("block_tables", block_tables), ("pad_lens", pad_lens)):
        if t.dtype != torch.int32:
            raise ValueError(f"{name} must be int32")
    c = cache.c_struct()
    ws_ptr = _ptr(workspace) if workspace is not None and workspace.numel() else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    check(native.lib().cb_padded_attention(
        _ptr(q), ctypes.byref(c), _ptr(cu_seqlens_q), _ptr(context_lens), _ptr(block_tables), _ptr(pad_lens),
        context_lens.shape[0], q.shape[0], block_tables.shape[1], max_q_len, max_context_len,
        float(scale), _ptr(out), ws_ptr, ws_bytes, _stream_handle(stream)), "cb_padded_attention")
    return out


def cb_attention_workspace_size_gqa(cache: KVCache, num_q_heads: int, num_seqs: int, num_tokens: int,
                                    max_context_len: int) -> int:
    c = cache.c_struct()
    return int(native.lib().cb_attention_workspace_size_gqa(ctypes.byref(c), num_q_heads, num_seqs, num_tokens,
                                                            max_context_len))


def cb_ragged_attention_gqa(q: torch.Tensor, cache: KVCache, cu_seqlens_q: torch.Tensor,
                            context_lens: torch.Tensor, block_tables: torch.Tensor, *,
                            max_q_len: int, max_context_len: int, scale: float, out: torch.Tensor,
                            workspace: Optional[torch.Tensor], stream=None) -> torch.Tensor:
    """cb_ragged_attention with q's heads (q.shape[1]) a multiple of the cache's."""
    for name, t in (("cu_seqlens_q", cu_seqlens_q), ("context_lens", context_lens),
                    ("block_tables", block_tables)):
        if t.dtype != torch.int32:
            raise ValueError(f"{name} must be int32")
    c = cache.c_struct()
    ws_ptr = _ptr(workspace) if workspace is not None and workspace.numel() else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    check(native.lib().cb_ragged_attention_gqa(
        _ptr(q), q.shape[1], ctypes.byref(c), _ptr(cu_seqlens_q), _ptr(context_lens), _ptr(block_tables),
        context_lens.shape[0], q.shape[0], block_tables.shape[1], max_q_len, max_context_len,
        float(scale), _ptr(out), ws_ptr, ws_bytes, _stream_handle(stream)), "cb_ragged_attention_gqa")
    return out


def cb_append_kv_dims(k_new: torch.Tensor, v_new: torch.Tensor, slot_mapping: torch.Tensor,
                      dims: torch.Tensor, cache: KVCache, stream=None) -> None:
    """cb_append_kv with the token count in dims[1] (device); k_new's rows bound it."""
    if slot_mapping.dtype != torch.int64 or dims.dtype != torch.int32:
        raise ValueError("slot_mapping must be int64 and dims int32")
    c = cache.c_struct()
    check(native.lib().cb_append_kv_dims(_ptr(k_new), _ptr(v_new), _ptr(slot_mapping), _ptr(dims),
                                         k_new.shape[0], ctypes.byref(c), _stream_handle(stream)),
          "cb_append_kv_dims")


def cb_plan_step(cache: KVCache, cu_seqlens_q: torch.Tensor, context_lens: torch.Tensor, *,
                 num_tokens: int, max_blocks_per_seq: int, max_q_len: int, max_context_len: int,
                 workspace: torch.Tensor, dims: Optional[torch.Tensor] = None,
                 num_q_heads: Optional[int] = None, stream=None) -> None:
    """Build the step's work lists in `workspace` (sizes are capacities when dims is given).
    num_q_heads: query heads of the planned calls when they differ from the
    cache's (grouped-query attention, cb_plan_step_gqa)."""
    for name, t in (("cu_seqlens_q", cu_seqlens_q), ("context_lens", context_lens)):
        if t.dtype != torch.int32:
            raise ValueError(f"{name} must be int32")
    c = cache.c_struct()
    rest = (_ptr(cu_seqlens_q), _ptr(context_lens), _ptr(dims), context_lens.shape[0], num_tokens,
            max_blocks_per_seq, max_q_len, max_context_len, _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream_handle(stream))
    if num_q_heads is None:
        check(native.lib().cb_plan_step(ctypes.byref(c), *rest), "cb_plan_step")
    else:
        check(native.lib().cb_plan_step_gqa(ctypes.byref(c), num_q_heads, *rest), "cb_plan_step_gqa")


def cb_ragged_attention_planned(q: torch.Tensor, cache: KVCache, cu_seqlens_q: torch.Tensor,
                                context_lens: torch.Tensor, block_tables: torch.Tensor, *,
                                max_q_len: int, max_context_len: int, scale: float, out: torch.Tensor,
                                workspace: torch.Tensor, dims: Optional[torch.Tensor] = None,
                                stream=None) -> torch.Tensor:
    """cb_ragged_attention over the plan cb_plan_step built in `workspace`.  When
    q has more heads than the cache (grouped-query attention) the call goes to
    cb_ragged_attention_planned_gqa, over a plan made with the same num_q_heads."""
    c = cache.c_struct()
    rest = (ctypes.byref(c), _ptr(cu_seqlens_q), _ptr(context_lens), _ptr(block_tables), _ptr(dims),
            context_lens.shape[0], q.shape[0], block_tables.shape[1], max_q_len, max_context_len, float(scale),
            _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(), _stream_handle(stream))
    if q.shape[1] == cache.num_heads:
        check(native.lib().cb_ragged_attention_planned(_ptr(q), *rest), "cb_ragged_attention_planned")
    else:
        check(native.lib().cb_ragged_attention_planned_gqa(_ptr(q), q.shape[1], *rest),
              "cb_ragged_attention_planned_gqa")
    return out


def cb_decode_attention_noalloc(q: torch.Tensor, cache: KVCache, cu_seqlens_q: torch.Tensor,
                                context_lens: torch.Tensor, block_tables: torch.Tensor, *,
                                max_context_len: int, scale: float, out: torch.Tensor,
                                stream=None) -> torch.Tensor:
    """Decode-only attention whose scratch is a fixed array the library reserves
    in device memory, for callers that cannot allocate or lend a workspace."""
    c = cache.c_struct()
    check(native.lib().cb_decode_attention_noalloc(
        _ptr(q), ctypes.byref(c), _ptr(cu_seqlens_q), _ptr(context_lens), _ptr(block_tables),
        context_lens.shape[0], q.shape[0], block_tables.shape[1], max_context_len, float(scale),
        _ptr(out), _stream_handle(stream)), "cb_decode_attention_noalloc")
    return out


def cb_check_device_errors(stream=None) -> None:
    check(native.lib().cb_check_device_errors(_stream_handle(stream)), "cb_check_device_errors")


def cb_synth_tokens(out: torch.Tensor, seed: int, kind: int, layer: int, seq_ids: torch.Tensor,
                    positions: torch.Tensor, stream=None) -> torch.Tensor:
    n, H, A = out.shape
    check(native.lib().cb_synth_tokens(_ptr(out), _DTYPES[out.dtype], seed, kind, layer,
                                       _ptr(seq_ids), _ptr(positions), n, H, A,
                                       _stream_handle(stream)), "cb_synth_tokens")
    return out


def cb_synth_fill_cache(pool: torch.Tensor, seed: int, kind: int, layer: int, seq_ids: torch.Tensor,
                        prefix_lens: torch.Tensor, block_tables: torch.Tensor, max_prefix: int,
                        stream=None) -> None:
    NB, H, B, A = pool.shape
    check(native.lib().cb_synth_fill_cache(
        _ptr(pool), _DTYPES[pool.dtype], seed, kind, layer, _ptr(seq_ids), _ptr(prefix_lens),
        _ptr(block_tables), block_tables.shape[0], block_tables.shape[1], NB, B, H, A, max_prefix,
        _stream_handle(stream)), "cb_synth_fill_cache")


# ---------------------------------------------------------------------------
# Host scheduler
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class Batch:
    """Copy of one cb_batch (numpy arrays)."""
    num_decode: int
    max_q_len: int
    max_context_len: int
    cu_seqlens_q: np.ndarray
    context_lens: np.ndarray
    block_tables: np.ndarray
    slot_mapping: np.ndarray
    request_ids: np.ndarray
    evicted_ids: np.ndarray
    preempted_ids: np.ndarray

    @property
    def num_seqs(self) -> int:
        return len(self.context_lens)

    @property
    def T(self) -> int:
        return int(self.cu_seqlens_q[-1])

    @property
    def q_lens(self) -> np.ndarray:
        return np.diff(self.cu_seqlens_q)


def _arr(ptr, n, dtype):
    if n == 0:
        return np.zeros(0, dtype=dtype)
    return np.ctypeslib.as_array(ptr, shape=(n,)).astype(dtype, copy=True)


class Scheduler:
    """cb_scheduler_* on the host (no GPU needed)."""

    def __init__(self, token_budget: int, block_size: int, num_blocks: int, max_num_seqs: int = 0,
                 admission: str = "reserve_lifetime"):
        self._L = native.lib()
        cfg = native.cb_sched_config(token_budget, block_size, num_blocks, max_num_seqs,
                                     native.ADMISSION[admission])
        h = ctypes.c_void_p()
        check(self._L.cb_scheduler_create(ctypes.byref(cfg), ctypes.byref(h)), "cb_scheduler_create")
        self._h = h

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            self._L.cb_scheduler_destroy(h)
            self._h = None

    def add_request(self, rid: int, arrival_step: int, prompt_len: int, output_len: int) -> None:
        check(self._L.cb_add_request(self._h, rid, arrival_step, prompt_len, output_len), "cb_add_request")

    def build_batch(self) -> Batch:
        b = native.cb_batch()
        check(self._L.cb_build_batch(self._h, ctypes.byref(b)), "cb_build_batch")
        S, T, W = b.num_seqs, b.num_tokens, b.max_blocks_per_seq
        return Batch(num_decode=b.num_decode, max_q_len=b.max_q_len, max_context_len=b.max_context_len,
                     cu_seqlens_q=_arr(b.cu_seqlens_q, S + 1, np.int32),
                     context_lens=_arr(b.context_lens, S, np.int32),
                     block_tables=_arr(b.block_tables, S * W, np.int32).reshape(S, W),
                     slot_mapping=_arr(b.slot_mapping, T, np.int64),
                     request_ids=_arr(b.request_ids, S, np.int64),
                     evicted_ids=_arr(b.evicted_ids, b.num_evicted, np.int64),
                     preempted_ids=_arr(b.preempted_ids, b.num_preempted, np.int64))

    def complete_step(self) -> None:
        check(self._L.cb_complete_step(self._h), "cb_complete_step")

    def stats(self) -> native.cb_sched_stats:
        s = native.cb_sched_stats()
        check(self._L.cb_scheduler_stats(self._h, ctypes.byref(s)), "cb_scheduler_stats")
        return s

    @property
    def idle(self) -> bool:
        s = self.stats()
        return s.num_waiting == 0 and s.num_running == 0
