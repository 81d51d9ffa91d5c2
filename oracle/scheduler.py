"""Iteration-level scheduler step (oracle; test infrastructure only).

Rules restated from

* Hugging Face blog "Continuous batching from first principles", section
  *Continuous batching*: aim for m tokens per batch; first add every request in
  its decoding phase at one token each; fill the rest with prompts in their
  prefill phase, chunked as needed; remove finished requests as soon as they
  are done and replace them with waiting ones (dynamic scheduling);
* hassanahmed.net, "How Continuous Batching Speeds Up LLM Serving", the
  scheduler loop: each pass first drops finished requests and releases their
  KV blocks, then admits the head of the waiting queue while it fits, then runs
  exactly one forward pass; and its paragraph on PagedAttention: the cache is
  handed out and reclaimed in fixed-size blocks;
* blog section *Attention*: the prefill pass over a prompt produces the first
  new token; each decode pass produces one more.

Readings where the pages leave the step open:

* admission is strict FIFO ordered by (arrival_step, id); the head is admitted
  iff it has arrived, the running set is below max_num_seqs (0 = no cap) and
  the unreserved blocks cover ceil((prompt_len + output_len) / B) -- the whole
  lifetime is reserved at admission, so a running request never runs short;
* decode tokens are taken in running (admission) order; if they exceed m the
  later ones wait;
* prefill room is filled greedily in running order, each request taking
  min(remaining prompt, room); a request admitted this step may prefill now;
* physical blocks are handed out lowest free id first, in batch order and
  position order, when a position first touches a new logical block;
* the batch lists decode sequences first, then prefill chunks;
* a request is finished when it has produced output_len tokens; it is evicted
  (its blocks freed) at the start of the next step.

Admission with preemption (admission="prompt_preempt"), hassanahmed.net, the
paragraph on the memory manager under continuous batching: when the card
fills, a request is evicted temporarily and brought back later.  Read as
preemption by recompute:

* the head is admitted when the free blocks cover its prefill, and those
  blocks are taken at once, lowest ids first;
* running requests take their decode blocks before anyone is admitted: when a
  decode token enters a new block and none is free, the most recently admitted
  running request is preempted, repeatedly, the decoding request itself last;
  a step that preempted admits no one;
* a preempted request gives back all its blocks, keeps the output tokens it
  produced, and rejoins the waiting queue at its (arrival, id) place -- the
  head, admission being FIFO; its next prefill covers prompt + generated
  tokens (every token it knows) and yields its next output token.
"""
from __future__ import annotations

import dataclasses
import heapq
import math
from typing import List, Optional

import numpy as np


@dataclasses.dataclass
class _Req:
    id: int
    arrival: int
    prompt_len: int
    output_len: int
    prefill_len: int = 0       # tokens of the next prefill (the prompt, or all known after preemption)
    computed: int = 0          # tokens whose K/V is in the cache
    generated: int = 0         # output tokens produced
    blocks: list = dataclasses.field(default_factory=list)
    reserved: int = 0


@dataclasses.dataclass
class Batch:
    request_ids: np.ndarray    # [S] int64
    q_lens: np.ndarray         # [S] int32
    cu_seqlens_q: np.ndarray   # [S+1] int32
    context_lens: np.ndarray   # [S] int32
    block_tables: np.ndarray   # [S, W] int32, -1 padded
    slot_mapping: np.ndarray   # [T] int64
    evicted_ids: np.ndarray    # [E] int64
    num_decode: int
    preempted_ids: np.ndarray = dataclasses.field(default_factory=lambda: np.zeros(0, np.int64))

    @property
    def num_seqs(self) -> int:
        return len(self.q_lens)

    @property
    def T(self) -> int:
        return int(self.cu_seqlens_q[-1])


class Scheduler:
    def __init__(self, token_budget: int, block_size: int, num_blocks: int, max_num_seqs: int = 0,
                 admission: str = "reserve_lifetime"):
        if token_budget < 1 or block_size < 1 or num_blocks < 1 or max_num_seqs < 0:
            raise ValueError("bad scheduler config")
        if admission not in ("reserve_lifetime", "prompt_preempt"):
            raise ValueError("unknown admission policy")
        self.preempting = admission == "prompt_preempt"
        self.num_preempted = 0
        self.recomputed_tokens = 0
        self.m = token_budget
        self.B = block_size
        self.NB = num_blocks
        self.max_num_seqs = max_num_seqs
        self.step = 0
        self.waiting: List[_Req] = []      # kept sorted by (arrival, id)
        self.running: List[_Req] = []      # admission order
        self.free = list(range(num_blocks))
        heapq.heapify(self.free)
        self.reserved_total = 0
        self.finished = 0
        self._pending: Optional[list] = None

    def _need(self, r: _Req) -> int:
        return math.ceil((r.prompt_len + r.output_len) / self.B)

    def add_request(self, rid: int, arrival_step: int, prompt_len: int, output_len: int) -> None:
        r = _Req(rid, arrival_step, prompt_len, output_len, prefill_len=prompt_len)
        if prompt_len < 1 or output_len < 1 or arrival_step < 0 or self._need(r) > self.NB:
            raise ValueError("request can never be admitted")
        self._enqueue(r)

    def _enqueue(self, r: _Req) -> None:
        key = (r.arrival, r.id)
        i = len(self.waiting)
        while i > 0 and (self.waiting[i - 1].arrival, self.waiting[i - 1].id) > key:
            i -= 1
        self.waiting.insert(i, r)

    def _preempt(self, r: _Req, preempted: list) -> None:
        for b in r.blocks:
            heapq.heappush(self.free, b)
        r.blocks = []
        self.recomputed_tokens += r.computed
        r.computed = 0
        r.prefill_len = r.prompt_len + r.generated
        self._enqueue(r)
        preempted.append(r.id)
        self.num_preempted += 1

    def build_batch(self) -> Batch:
        if self._pending is not None:
            raise RuntimeError("previous batch not completed")
        # 1. evict finished requests, give their blocks back
        evicted = []
        keep = []
        for r in self.running:
            if r.generated == r.output_len:
                evicted.append(r.id)
                for b in r.blocks:
                    heapq.heappush(self.free, b)
                self.reserved_total -= r.reserved
                self.finished += 1
            else:
                keep.append(r)
        self.running = keep
        room = self.m
        chosen = []                       # (request, n_tokens, is_decode)
        preempted = []

        def admit():                      # 2. admit from the FIFO head while it fits
            while self.waiting:
                r = self.waiting[0]
                if r.arrival > self.step:
                    break
                if self.max_num_seqs and len(self.running) >= self.max_num_seqs:
                    break
                if self.preempting:
                    need = math.ceil(r.prefill_len / self.B)
                    if len(self.free) < need:
                        break
                    self.waiting.pop(0)
                    r.blocks = [heapq.heappop(self.free) for _ in range(need)]
                else:
                    need = self._need(r)
                    if self.NB - self.reserved_total < need:
                        break
                    self.waiting.pop(0)
                    r.reserved = need
                    self.reserved_total += need
                self.running.append(r)

        def choose_decodes():             # 3. decode requests first, one token each
            nonlocal room
            i = 0
            while i < len(self.running) and room > 0:
                r = self.running[i]
                i += 1
                if r.computed < r.prefill_len:
                    continue
                if self.preempting and r.computed // self.B >= len(r.blocks):
                    while not self.free and self.running[-1] is not r:
                        self._preempt(self.running.pop(), preempted)
                    if not self.free:
                        self._preempt(self.running.pop(), preempted)
                        break
                    r.blocks.append(heapq.heappop(self.free))
                chosen.append((r, 1, True))
                room -= 1

        if self.preempting:
            choose_decodes()
            if not preempted:
                admit()
        else:
            admit()
            choose_decodes()
        num_decode = len(chosen)
        # 4. then prefill chunks, greedily in admission order
        for r in self.running:
            if r.computed < r.prefill_len and room > 0:
                n = min(r.prefill_len - r.computed, room)
                chosen.append((r, n, False))
                room -= n
        # 5. blocks for the new positions, 6. metadata
        S = len(chosen)
        q_lens = np.array([n for _, n, _ in chosen], dtype=np.int32)
        cu = np.zeros(S + 1, dtype=np.int32)
        cu[1:] = np.cumsum(q_lens)
        slots = np.empty(int(cu[-1]), dtype=np.int64)
        for s, (r, n, _) in enumerate(chosen):
            for k in range(n):
                pos = r.computed + k
                if pos // self.B >= len(r.blocks):
                    r.blocks.append(heapq.heappop(self.free))
                slots[cu[s] + k] = r.blocks[pos // self.B] * self.B + pos % self.B
        W = max((len(r.blocks) for r, _, _ in chosen), default=0)
        bt = np.full((S, W), -1, dtype=np.int32)
        for s, (r, _, _) in enumerate(chosen):
            bt[s, :len(r.blocks)] = r.blocks
        ctx = np.array([r.computed + n for r, n, _ in chosen], dtype=np.int32)
        self._pending = chosen
        return Batch(request_ids=np.array([r.id for r, _, _ in chosen], dtype=np.int64),
                     q_lens=q_lens, cu_seqlens_q=cu, context_lens=ctx, block_tables=bt,
                     slot_mapping=slots, evicted_ids=np.array(evicted, dtype=np.int64),
                     num_decode=num_decode, preempted_ids=np.array(preempted, dtype=np.int64))

    def complete_step(self) -> None:
        if self._pending is None:
            raise RuntimeError("no batch to complete")
        for r, n, is_decode in self._pending:
            r.computed += n
            if is_decode or r.computed == r.prefill_len:
                r.generated += 1
        self._pending = None
        self.step += 1

    @property
    def idle(self) -> bool:
        """No request waiting and none running (finished ones already evicted)."""
        return not self.waiting and not self.running
