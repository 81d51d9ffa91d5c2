"""CPU oracle for the ragged continuous-batching attention step.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this package:
only the tests, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may use it.  It shares no code with
the CUDA library and imports nothing from it.

Contents (each function cites the passage it restates):

* ``attention``  -- masked softmax attention per sequence, unpacked, in fp64
  (Hugging Face blog "Continuous batching from first principles", sections
  *Attention*, *KV-cache*, *Chunked prefill*, *Continuous batching*; page
  "continuous-batching" (zhangchitc.github.io), section "Ragged batching:
  attention in per-request blocks").
* ``kv_cache``   -- where the step's new keys/values land in a block-paged
  cache, and reading a sequence's history back out of one (page
  "continuous-batching", section "Inside the kernel: cu_seqlens splits six
  rows back into three"; hassanahmed.net "How Continuous Batching Speeds Up
  LLM Serving", paragraph on PagedAttention's fixed-size blocks).
* ``scheduler``  -- the iteration-level scheduler step: evict, admit, decode
  first, fill the token budget with chunked prefill (blog section
  *Continuous batching*, the three-item rule and "Dynamic scheduling";
  hassanahmed.net, the evict/admit/step loop).

Parity pins: every function here is pinned by ``tests/test_oracle_*.py``
against closed forms, library routines, hand-derived fixtures under
``tests/golden/`` and invariants the pages state.  No function is unpinned.
"""
from . import attention, kv_cache, scheduler  # noqa: F401
