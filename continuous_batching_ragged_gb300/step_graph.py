"""A whole multi-layer step captured once as a CUDA graph and replayed.

Hugging Face blog "Continuous batching from first principles", section
"Continuous batching": every layer of a step runs on the same packed batch,
and fixed shapes are what make a step capturable as a CUDA graph.  Here the
shapes are fixed by capacity: the step's metadata lives in device buffers of
fixed size and address, its sizes in a device `dims` array, and every launch
of the step (one plan, then per layer cb_append_kv_dims and
cb_ragged_attention_planned) has the same arguments from step to step.  A step
is then: copy the new metadata into the buffers (two host-to-device copies),
replay the graph.

This module is host plumbing over the C ABI: buffer management, the staging
copy and the capture.  Every step of the computation runs in the library's
kernels.
"""
from __future__ import annotations

from typing import List, Optional

import numpy as np
import torch

from . import api


class StepGraph:
    """Capacity buffers, a captured graph of `len(caches)` layers, and replay.

    q, k_new, v_new: one [max_tokens, H, A] tensor per layer; the caller fills
    their first T rows before each replay.  outs: one [max_tokens, H, A]
    tensor per layer (or a single shared one) that receives each layer's rows.
    q and outs may carry more heads than the caches (grouped-query attention:
    a multiple of them); k_new and v_new carry the caches' heads.
    """

    def __init__(self, caches: List[api.KVCache], q: List[torch.Tensor], k_new: List[torch.Tensor],
                 v_new: List[torch.Tensor], outs: List[torch.Tensor], *, max_seqs: int,
                 max_blocks_per_seq: int, scale: float):
        if not (len(caches) == len(q) == len(k_new) == len(v_new)) or len(outs) not in (1, len(caches)):
            raise ValueError("one q, k_new, v_new per layer; one shared out or one per layer")
        self.caches, self.q, self.k_new, self.v_new = caches, q, k_new, v_new
        self.outs = outs if len(outs) == len(caches) else outs * len(caches)
        self.max_seqs = max_seqs
        self.max_tokens = q[0].shape[0]
        self.max_blocks = max_blocks_per_seq
        self.max_context = max_blocks_per_seq * caches[0].block_size
        self.scale = scale
        self.num_q_heads = q[0].shape[1]
        self.grouped = self.num_q_heads != caches[0].num_heads
        S, W = max_seqs, max_blocks_per_seq
        # int32 metadata, one buffer: dims[4] | cu[S+1] | context_lens[S] | block_tables[S*W]
        n = 4 + (S + 1) + S + S * W
        self._meta_dev = torch.zeros(n, dtype=torch.int32, device="cuda")
        self._meta_host = torch.zeros(n, dtype=torch.int32).pin_memory()
        self._slots_dev = torch.full((self.max_tokens,), -1, dtype=torch.int64, device="cuda")
        self._slots_host = torch.full((self.max_tokens,), -1, dtype=torch.int64).pin_memory()
        o = [0, 4, 4 + S + 1, 4 + 2 * S + 1, n]
        self.dims, self.cu, self.ctx = (self._meta_dev[o[i]:o[i + 1]] for i in range(3))
        self.block_tables = self._meta_dev[o[3]:o[4]].view(S, W)
        self._hv = [self._meta_host.numpy()[o[i]:o[i + 1]] for i in range(4)]
        ws = (api.cb_attention_workspace_size_gqa(caches[0], self.num_q_heads, S, self.max_tokens, self.max_context)
              if self.grouped else api.cb_attention_workspace_size(caches[0], S, self.max_tokens, self.max_context))
        self.workspace = torch.empty(ws, dtype=torch.uint8, device="cuda")
        self.graph: Optional[torch.cuda.CUDAGraph] = None
        self.num_tokens = 0

    def load(self, cu_seqlens_q: np.ndarray, context_lens: np.ndarray, block_tables: np.ndarray,
             slot_mapping: np.ndarray, max_q_len: int, max_context_len: int, stream=None) -> None:
        """Stage one step's metadata and copy it to the device buffers (stream-ordered)."""
        S, T = len(context_lens), len(slot_mapping)
        W = block_tables.shape[1] if block_tables.ndim == 2 else 0
        if S > self.max_seqs or T > self.max_tokens or W > self.max_blocks or max_context_len > self.max_context:
            raise ValueError("step exceeds the graph's capacities")
        dims, cu, ctx, bt = self._hv
        dims[:] = (S, T, max_q_len, max_context_len)
        cu[:S + 1] = cu_seqlens_q
        ctx[:S] = context_lens
        bt.reshape(self.max_seqs, self.max_blocks)[:S, :W] = block_tables
        self._slots_host.numpy()[:T] = slot_mapping
        s = stream if stream is not None else torch.cuda.current_stream()
        with torch.cuda.stream(s):
            self._meta_dev.copy_(self._meta_host, non_blocking=True)
            self._slots_dev.copy_(self._slots_host, non_blocking=True)
        self.num_tokens = T

    def _step(self) -> None:
        kw = dict(num_tokens=self.max_tokens, max_blocks_per_seq=self.max_blocks,
                  max_q_len=self.max_tokens, max_context_len=self.max_context)
        api.cb_plan_step(self.caches[0], self.cu, self.ctx, workspace=self.workspace, dims=self.dims,
                         num_q_heads=self.num_q_heads if self.grouped else None, **kw)
        for layer, cache in enumerate(self.caches):
            api.cb_append_kv_dims(self.k_new[layer], self.v_new[layer], self._slots_dev, self.dims, cache)
            api.cb_ragged_attention_planned(
                self.q[layer], cache, self.cu, self.ctx, self.block_tables, dims=self.dims,
                max_q_len=self.max_tokens, max_context_len=self.max_context, scale=self.scale,
                out=self.outs[layer], workspace=self.workspace)

    def run_eager(self) -> None:
        """The same launches without a graph (also resolves per-device state before a capture)."""
        self._step()

    def capture(self) -> None:
        """Capture the step once.  Run one eager step (run_eager) first."""
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self._step()

    def replay(self) -> None:
        if self.graph is None:
            raise RuntimeError("capture() first")
        self.graph.replay()
