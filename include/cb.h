/*
 * cb.h -- C ABI of the ragged continuous-batching attention step on one GPU.
 *
 * One step of continuous batching, as these pages define it:
 *
 *   - Hugging Face blog "Continuous batching from first principles", section
 *     "Continuous batching": sequences are concatenated without padding
 *     ("ragged batching"); each step holds at most m tokens, decoding requests
 *     first at one token each, the rest filled by chunked prefill; finished
 *     requests leave and waiting ones join.
 *   - page "continuous-batching" (zhangchitc.github.io), section "Inside the
 *     kernel: cu_seqlens splits six rows back into three": the step's keys and
 *     values are written into each request's cache entry, then every key and
 *     value of the request is read back block by block for attention, with an
 *     online softmax; cu_seqlens delimits each request's rows.
 *
 * Conventions for every entry point
 *   - Device buffers are allocated and owned by the caller.  The library keeps
 *     no pointer after a call returns.  Attention needs a caller-provided
 *     workspace (cb_attention_workspace_size).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Device work is enqueued on it and the call returns after the launch.
 *   - Errors that can be seen on the host (null pointers, sizes, unsupported
 *     dtype/shape combinations, bounds given by the caller) are returned before
 *     anything is launched.  Errors that only the device can see (a slot or
 *     block id outside the pool, metadata that contradicts the host bounds, a
 *     bounded wait that ran out) set a per-device error word instead: the
 *     offending work item is skipped and cb_check_device_errors reports it.
 *   - No C++ exception crosses the ABI.  cb_last_error() describes the most
 *     recent failure of a call made on the calling thread.
 *   - Head-major paged cache: K and V are separate pools, each
 *     [num_blocks][num_heads][block_size][head_dim], row-major.  Token slot
 *     s = block_id * block_size + offset lives at pool[block_id][h][offset][:].
 *     Packed token tensors (q, k_new, v_new, out) are [num_tokens][num_heads]
 *     [head_dim], row-major.
 */
#ifndef CB_H_
#define CB_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CB_OK = 0,
  CB_ERR_INVALID = 1,      /* bad argument or metadata */
  CB_ERR_BOUNDS = 2,       /* a slot or block id outside the pool (device) */
  CB_ERR_NO_BLOCKS = 3,    /* scheduler: request can never fit the pool */
  CB_ERR_TIMEOUT = 4,      /* a bounded device wait ran out (device) */
  CB_ERR_CUDA = 5,         /* a CUDA runtime call failed */
  CB_ERR_UNSUPPORTED = 6   /* dtype / head_dim / block_size combination not built */
} cb_status;

typedef enum { CB_DTYPE_F32 = 0, CB_DTYPE_BF16 = 1 } cb_dtype;

/* One layer's paged KV cache.  k and v point to device pools of
 * num_blocks * num_heads * block_size * head_dim elements of `dtype`, each
 * 16-byte aligned.  Caller-owned. */
typedef struct {
  void* k;
  void* v;
  int32_t num_blocks;
  int32_t block_size;
  int32_t num_heads;
  int32_t head_dim;
  cb_dtype dtype;
} cb_kv_cache;

/* ---------------------------------------------------------------------------
 * cb_append_kv -- write this step's keys and values into the cache.
 * Page "continuous-batching" (zhangchitc.github.io), section "Inside the
 * kernel": a step first stores every new key and value row under the request
 * it belongs to; attention then reads the cache.
 *
 *   k_new, v_new  device [num_tokens][num_heads][head_dim] of cache->dtype,
 *                 16-byte aligned.
 *   slot_mapping  device int64 [num_tokens]; token t goes to slot
 *                 slot_mapping[t]; a negative slot skips the token.
 *   A slot >= num_blocks * block_size sets CB_ERR_BOUNDS on the device word and
 *   is not written.  head_dim * element size must be a multiple of 16 bytes.
 * ------------------------------------------------------------------------- */
cb_status cb_append_kv(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                       int32_t num_tokens, const cb_kv_cache* cache, void* stream);

/* ---------------------------------------------------------------------------
 * cb_ragged_attention -- attention of one packed, padding-free step.
 * Hugging Face blog "Continuous batching from first principles", sections
 * "Attention" (masked row-wise softmax of Q K^T times V), "Chunked prefill"
 * (a chunk sees the cached keys of its earlier tokens plus itself, causally)
 * and "Continuous batching" (concatenated sequences never see each other);
 * page "continuous-batching", section "Ragged batching" (a decoding request's
 * one query against all of its keys, a prefilling request's causal block).
 *
 * Sequence s owns packed rows cu_seqlens_q[s] .. cu_seqlens_q[s+1]-1 (q_len_s
 * >= 1 rows) and has context_lens[s] keys in the cache AFTER this step's
 * append, so p_s = context_lens[s] - q_len_s were cached before the step.
 * Its row i (0-based) attends keys j = 0 .. p_s + i:
 *     out = softmax_j(scale * q . k_j) v_j,   accumulated in fp32.
 *
 *   q             device [num_tokens][H][A] of cache->dtype.
 *   cu_seqlens_q  device int32 [num_seqs + 1], cu[0] = 0, cu[num_seqs] = num_tokens.
 *   context_lens  device int32 [num_seqs].
 *   block_tables  device int32 [num_seqs][max_blocks_per_seq]; logical block b
 *                 of sequence s is physical block block_tables[s][b].  Entries
 *                 past ceil(context_lens[s] / block_size) are never read.
 *   max_q_len, max_context_len  host upper bounds over the batch; the device
 *                 flags (CB_ERR_INVALID) and skips any sequence exceeding them.
 *   out           device [num_tokens][H][A] of cache->dtype; every row written.
 *   workspace     device scratch of at least cb_attention_workspace_size(...)
 *                 bytes, 256-byte aligned: the step's work lists, split-KV
 *                 decode partials, and (bf16, when num_tokens > num_seqs and
 *                 max_context_len > 2048) 136 MB of partial rows for prefill
 *                 pairs cut into KV segments; its contents need no
 *                 initialisation and are not preserved.
 *   Concurrent calls must not share one workspace.
 * Built combinations: bf16 with head_dim 128 and block_size in {8,16,32,64,128}
 * (prefill chunks on tcgen05 tensor cores, decode rows split-KV on CUDA cores);
 * f32 with head_dim 64 or 128 and any block_size (every row on CUDA cores).
 * ------------------------------------------------------------------------- */
size_t cb_attention_workspace_size(const cb_kv_cache* cache, int32_t num_seqs,
                                   int32_t num_tokens, int32_t max_context_len);

cb_status cb_ragged_attention(const void* q, const cb_kv_cache* cache,
                              const int32_t* cu_seqlens_q, const int32_t* context_lens,
                              const int32_t* block_tables, int32_t num_seqs, int32_t num_tokens,
                              int32_t max_blocks_per_seq, int32_t max_q_len,
                              int32_t max_context_len, float scale, void* out,
                              void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Grouped-query attention (GQA / MQA): fewer key/value heads than query heads.
 * The pages have no counterpart; every page assumes one key/value head per
 * query head.  Here q and out have num_q_heads heads, the cache (and k_new,
 * v_new of cb_append_kv) cache->num_heads = H_kv heads, num_q_heads a
 * multiple of H_kv, and query head h attends with key/value head
 * h / (num_q_heads / H_kv) (groups of consecutive query heads).  Otherwise
 * identical to cb_ragged_attention, which is the case num_q_heads = H_kv.
 * Decode rows of a group run on one of two kernels: CUDA cores, a unit
 * covering up to four query heads of one group, or tensor cores (head_dim
 * 128, groups of 4 to 32 heads), a unit covering the whole group; either way
 * each K/V byte read from memory serves all the unit's heads.  Groups of more
 * than four take the tensor cores; groups of four take them too except in
 * decode-only steps with at least 10 (sequence, key/value head) units per SM
 * given on the host (dims NULL).  The two kernels agree within fp32
 * accumulation rounding, not bit for bit, so a step of groups of four can
 * differ in its last bits between a host-sized call and a dims call.
 * Grouped heads need bf16 and a block size that is a multiple of 16
 * (CB_ERR_UNSUPPORTED otherwise); the workspace must be
 * cb_attention_workspace_size_gqa bytes.
 * ------------------------------------------------------------------------- */
size_t cb_attention_workspace_size_gqa(const cb_kv_cache* cache, int32_t num_q_heads,
                                       int32_t num_seqs, int32_t num_tokens, int32_t max_context_len);
cb_status cb_ragged_attention_gqa(const void* q, int32_t num_q_heads, const cb_kv_cache* cache,
                                  const int32_t* cu_seqlens_q, const int32_t* context_lens,
                                  const int32_t* block_tables, int32_t num_seqs, int32_t num_tokens,
                                  int32_t max_blocks_per_seq, int32_t max_q_len,
                                  int32_t max_context_len, float scale, void* out,
                                  void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Planned steps and CUDA-graph capture.
 * Hugging Face blog "Continuous batching from first principles", section
 * "Continuous batching": every layer of a step sees the same packed batch, and
 * static shapes are what let a step be captured as a CUDA graph.  So the work
 * lists are built once per step (cb_plan_step) and every layer's attention
 * reuses them (cb_ragged_attention_planned); with `dims` set, every launch of
 * a step has the same shape and arguments from step to step, so a step made
 * of these calls can be captured once and replayed with new metadata.
 *
 *   dims  NULL, or device int32[4] = {num_seqs, num_tokens, max_q_len,
 *         max_context_len} of the step.  When set, the host arguments of the
 *         same names are CAPACITIES: the extents the metadata buffers, q, out,
 *         k_new, v_new and slot_mapping are allocated for (block_tables is
 *         [num_seqs capacity][max_blocks_per_seq]).  A step whose device sizes
 *         exceed them sets CB_ERR_INVALID on the device word and runs empty.
 *   Only bf16 caches with head_dim 128 and a block size that is a multiple of
 *   16 are planned (CB_ERR_UNSUPPORTED otherwise).
 *   Make one call of each outside stream capture first: it resolves
 *   per-device state (the error word, kernel attributes, a second stream).
 * ------------------------------------------------------------------------- */

/* cb_append_kv with the token count read from dims[1] on the device;
 * max_tokens bounds it (the extent of k_new, v_new and slot_mapping). */
cb_status cb_append_kv_dims(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                            const int32_t* dims, int32_t max_tokens, const cb_kv_cache* cache,
                            void* stream);

/* Build the step's work lists in `workspace` (at least
 * cb_attention_workspace_size(cache, num_seqs, num_tokens, max_context_len)
 * bytes) from cu_seqlens_q and context_lens.  Reads only the metadata;
 * cache supplies the shape (its pools may be NULL).  The lists stay valid
 * until the metadata changes or the workspace is reused for anything else. */
cb_status cb_plan_step(const cb_kv_cache* cache, const int32_t* cu_seqlens_q,
                       const int32_t* context_lens, const int32_t* dims, int32_t num_seqs,
                       int32_t num_tokens, int32_t max_blocks_per_seq, int32_t max_q_len,
                       int32_t max_context_len, void* workspace, size_t workspace_bytes,
                       void* stream);

/* cb_ragged_attention over the plan that cb_plan_step built in `workspace`:
 * same result, for any layer's q, cache pools and out.  cu_seqlens_q,
 * context_lens, dims, the sizes, the cache shape and workspace_bytes must be
 * the ones the plan was made with (CB_ERR_INVALID otherwise).  Calls over one
 * plan must not overlap on the GPU (they share its claim counters). */
cb_status cb_ragged_attention_planned(const void* q, const cb_kv_cache* cache,
                                      const int32_t* cu_seqlens_q, const int32_t* context_lens,
                                      const int32_t* block_tables, const int32_t* dims,
                                      int32_t num_seqs, int32_t num_tokens,
                                      int32_t max_blocks_per_seq, int32_t max_q_len,
                                      int32_t max_context_len, float scale, void* out,
                                      void* workspace, size_t workspace_bytes, void* stream);

/* The same two calls for grouped-query attention: q and out carry num_q_heads
 * heads (a positive multiple of the cache's heads), as in
 * cb_ragged_attention_gqa; the workspace is sized by
 * cb_attention_workspace_size_gqa.  A plan made by cb_plan_step_gqa serves
 * only cb_ragged_attention_planned_gqa calls with the same num_q_heads
 * (CB_ERR_INVALID otherwise). */
cb_status cb_plan_step_gqa(const cb_kv_cache* cache, int32_t num_q_heads, const int32_t* cu_seqlens_q,
                           const int32_t* context_lens, const int32_t* dims, int32_t num_seqs,
                           int32_t num_tokens, int32_t max_blocks_per_seq, int32_t max_q_len,
                           int32_t max_context_len, void* workspace, size_t workspace_bytes,
                           void* stream);
cb_status cb_ragged_attention_planned_gqa(const void* q, int32_t num_q_heads, const cb_kv_cache* cache,
                                          const int32_t* cu_seqlens_q, const int32_t* context_lens,
                                          const int32_t* block_tables, const int32_t* dims,
                                          int32_t num_seqs, int32_t num_tokens,
                                          int32_t max_blocks_per_seq, int32_t max_q_len,
                                          int32_t max_context_len, float scale, void* out,
                                          void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * cb_padded_attention -- attention of a left-padded rectangular batch, the
 * padded batching that ragged batching replaces.
 * Hugging Face blog "Continuous batching from first principles", section
 * "Continuous batching": without ragged batching, the sequences of a batch
 * are padded on the left to one common length and an attention mask keeps
 * the pad positions out of the softmax; inserting an n-token prompt into a
 * batch of B decoding sequences costs (n - 1)(B - 1) pad tokens.
 *
 * Same arguments and layout as cb_ragged_attention, plus
 *   pad_lens  device int32 [num_seqs]: the first pad_lens[s] rows of
 *             sequence s's chunk are padding (their K/V were appended like
 *             any other token).  With p_s = context_lens[s] - q_len_s, real
 *             row i (pad_lens[s] <= i < q_len_s) attends keys 0 .. p_s - 1 and
 *             p_s + pad_lens[s] .. p_s + i: the pad keys are masked out of
 *             every row.  The pad rows' own output rows are not written.
 * Needs a bf16 cache (CB_ERR_UNSUPPORTED otherwise) and
 * 0 <= pad_lens[s] < q_len_s; a sequence breaking that is left out and
 * reported as CB_ERR_INVALID by cb_check_device_errors.  Rows are computed at
 * the padded batch's full cost: every pad row and pad key goes through the
 * same kernels as real ones.
 * ------------------------------------------------------------------------- */
cb_status cb_padded_attention(const void* q, const cb_kv_cache* cache, const int32_t* cu_seqlens_q,
                              const int32_t* context_lens, const int32_t* block_tables,
                              const int32_t* pad_lens, int32_t num_seqs, int32_t num_tokens,
                              int32_t max_blocks_per_seq, int32_t max_q_len, int32_t max_context_len,
                              float scale, void* out, void* workspace, size_t workspace_bytes,
                              void* stream);

/* ---------------------------------------------------------------------------
 * cb_decode_attention_noalloc -- decode attention that allocates nothing.
 * The sources have no counterpart: this is a deployment variant of the decode
 * rows of cb_ragged_attention for callers that cannot allocate device memory
 * and have no workspace to lend -- for example an op running inside a host
 * framework whose caching allocator (or a KV pool sized to fill the GPU)
 * already owns all device memory, behind a plugin interface that passes only
 * the op's inputs and outputs.
 *
 * Same arguments and result as cb_ragged_attention for a step in which every
 * sequence has exactly one query token (num_tokens == num_seqs, max_q_len 1),
 * without the workspace.  The split-KV scratch lives instead in one array of
 * CB_NOALLOC_SCRATCH_BYTES that the library reserves in device memory on every
 * GPU that loads it, until the process exits.  A step whose scratch would not
 * fit (the size cb_attention_workspace_size reports for it) is rejected with
 * CB_ERR_INVALID before anything is launched.
 *   - The first call on a device looks up the array's device address with that
 *     device current; make that first call before any stream capture.
 *   - Every call shares the one array and it keeps the last call's contents;
 *     the call clears what must start at zero itself.  Calls whose GPU work
 *     overlaps (several streams or host threads) race on it and corrupt each
 *     other's results: serialise them, e.g. on one stream.
 *   - It calls no cudaMalloc, cudaFree or other allocating routine.
 * ------------------------------------------------------------------------- */
#define CB_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
cb_status cb_decode_attention_noalloc(const void* q, const cb_kv_cache* cache,
                                      const int32_t* cu_seqlens_q, const int32_t* context_lens,
                                      const int32_t* block_tables, int32_t num_seqs,
                                      int32_t num_tokens, int32_t max_blocks_per_seq,
                                      int32_t max_context_len, float scale, void* out,
                                      void* stream);

/* ---------------------------------------------------------------------------
 * Host scheduler: one iteration-level step at a time.
 * hassanahmed.net "How Continuous Batching Speeds Up LLM Serving", the
 * scheduler loop: drop finished requests and release their KV blocks, admit
 * waiting requests while they fit, run exactly one forward pass; Hugging Face
 * blog, section "Continuous batching": budget of m tokens, decoding requests
 * first at one token each, the remaining room filled by chunked prefill.
 *
 * Rules where the pages leave the step open: waiting requests are ordered by
 * (arrival_step, id) and admitted strictly FIFO when arrived, under
 * max_num_seqs (0 = no cap) and with ceil((prompt_len + output_len) /
 * block_size) unreserved blocks (the whole lifetime is reserved at admission);
 * decode tokens go in admission order; prefill room is filled greedily in
 * admission order; blocks are handed out lowest free id first; a request is
 * finished after output_len tokens (the prefill pass yields the first) and is
 * evicted at the start of the next cb_build_batch.
 *
 * Preemption (CB_ADMIT_PROMPT_PREEMPT).  hassanahmed.net, the paragraph on the
 * memory manager under continuous batching: when the card fills, a request
 * is evicted for a while and brought back later.  Read here as preemption by
 * recompute, with these rules:
 *   - The head of the queue is admitted when the free blocks cover its prefill.
 *     Those blocks are taken at once (lowest ids first).
 *   - When a decode token of request r needs a new block and none is free,
 *     the most recently admitted running request is preempted, repeatedly,
 *     until a block is free (r itself last).
 *   - A preempted request gives back all its blocks and keeps the output
 *     tokens it has produced. It rejoins the waiting queue at its original
 *     (arrival_step, id) place, which is the head, since admission is FIFO.
 *   - Its next prefill covers prompt_len + generated tokens, all of its known
 *     tokens, and yields its next output token.
 * The preempted ids of a step are reported in its batch.
 * ------------------------------------------------------------------------- */
typedef enum {
  /* reserve ceil((prompt_len + output_len) / block_size) blocks at admission:
   * a running request never runs short and is never preempted */
  CB_ADMIT_RESERVE_LIFETIME = 0,
  /* take the prompt's blocks at admission and one more block whenever a
   * decode token enters a new block; when none is free, preempt (below) */
  CB_ADMIT_PROMPT_PREEMPT = 1
} cb_admission;

typedef struct {
  int32_t token_budget;   /* m = max tokens per step (max_num_batched_tokens) */
  int32_t block_size;
  int32_t num_blocks;
  int32_t max_num_seqs;   /* 0 = unlimited */
  int32_t admission;      /* cb_admission; 0 (zero-initialised) = reserve the lifetime */
} cb_sched_config;

typedef struct cb_scheduler cb_scheduler;

/* Host arrays owned by the scheduler, valid until its next cb_build_batch or
 * cb_scheduler_destroy.  Sequences are listed decode first, then prefill. */
typedef struct {
  int32_t num_seqs;
  int32_t num_tokens;           /* T = sum of q_lens <= token_budget */
  int32_t num_decode;           /* the first num_decode sequences have q_len 1 */
  int32_t max_blocks_per_seq;   /* row stride of block_tables */
  int32_t max_q_len;
  int32_t max_context_len;
  const int32_t* cu_seqlens_q;  /* [num_seqs + 1] */
  const int32_t* context_lens;  /* [num_seqs] */
  const int32_t* block_tables;  /* [num_seqs][max_blocks_per_seq], -1 padded */
  const int64_t* slot_mapping;  /* [num_tokens] */
  const int64_t* request_ids;   /* [num_seqs] */
  int32_t num_evicted;
  const int64_t* evicted_ids;   /* [num_evicted], evicted by this call */
  int32_t num_preempted;
  const int64_t* preempted_ids; /* [num_preempted], preempted by this call (back to waiting) */
} cb_batch;

typedef struct {
  int64_t step;                 /* completed steps */
  int32_t num_waiting;
  int32_t num_running;          /* includes finished requests not yet evicted */
  int32_t free_blocks;
  int32_t reserved_blocks;
  int64_t num_finished;         /* evicted so far */
  int64_t num_preempted;        /* preemptions so far */
  int64_t recomputed_tokens;    /* prefill tokens spent re-computing preempted requests */
} cb_sched_stats;

cb_status cb_scheduler_create(const cb_sched_config* config, cb_scheduler** out);
void cb_scheduler_destroy(cb_scheduler* sched);
/* CB_ERR_NO_BLOCKS if the request could never be admitted (needs more blocks
 * than the pool holds); CB_ERR_INVALID for prompt_len < 1, output_len < 1,
 * arrival_step < 0 or an id already known. */
cb_status cb_add_request(cb_scheduler* sched, int64_t id, int64_t arrival_step,
                         int32_t prompt_len, int32_t output_len);
/* Evict, admit, choose this step's tokens, allocate blocks, emit metadata.
 * CB_ERR_INVALID if the previous batch was not completed. */
cb_status cb_build_batch(cb_scheduler* sched, cb_batch* out);
/* Account the last batch as run: cached tokens, output tokens, the clock. */
cb_status cb_complete_step(cb_scheduler* sched);
cb_status cb_scheduler_stats(const cb_scheduler* sched, cb_sched_stats* out);

/* ---------------------------------------------------------------------------
 * Errors.
 * cb_check_device_errors synchronises `stream`, reads and clears the current
 * device's error word and returns CB_ERR_TIMEOUT, CB_ERR_BOUNDS or
 * CB_ERR_INVALID (in that order of precedence) if any was raised since the
 * last check, else CB_OK.
 * ------------------------------------------------------------------------- */
cb_status cb_check_device_errors(void* stream);
const char* cb_last_error(void);

/* ---------------------------------------------------------------------------
 * cb_selftest_bounded_wait -- failure-detection self test.
 * Not a step of the method: launches one CTA that waits, with the same
 * bounded mbarrier wait the kernels use for every pipeline hand-off, on a
 * barrier nothing ever arrives at.  After timeout_ms (1..10000) the wait gives
 * up, the CTA sets CB_ERR_TIMEOUT on the device error word and exits, so the
 * context stays usable; cb_check_device_errors then returns CB_ERR_TIMEOUT.
 * ------------------------------------------------------------------------- */
cb_status cb_selftest_bounded_wait(int32_t timeout_ms, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* CB_H_ */
