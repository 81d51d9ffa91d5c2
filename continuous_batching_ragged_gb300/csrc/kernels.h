// Internal launch interface between the entry point and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "cb.h"

namespace cb {

struct AttnArgs {
  const void* q;
  void* out;
  const void* k_pool;
  const void* v_pool;
  const int32_t* cu_seqlens_q;
  const int32_t* context_lens;
  const int32_t* block_tables;
  int32_t num_seqs;
  int32_t num_tokens;
  int32_t max_blocks_per_seq;
  int32_t num_blocks;
  int32_t block_size;
  int32_t num_heads;      // query heads (q and out rows)
  int32_t num_kv_heads;   // heads of the cache pools; num_heads is a multiple of it
  int32_t head_dim;
  int32_t max_q_len;
  int32_t max_context_len;
  float scale_log2;       // softmax scale * log2(e)
  cb_dtype dtype;
  unsigned* err;
  // Device step sizes (num_seqs, num_tokens, max_q_len, max_context_len), or
  // null.  When set, the four host sizes above are capacities: buffer extents
  // that bound the device values, which only the step plan reads.
  const int32_t* dims = nullptr;
  // Left padding (cb_padded_attention), or null: the first pad_lens[s] rows
  // of sequence s's chunk are padding, their keys (positions p_s ..
  // p_s + pad - 1) are masked out of every row and their rows are not
  // written.  0 <= pad < q_len (the plan leaves a row out otherwise).
  const int32_t* pad_lens = nullptr;
};

// Keys per split of the register split-KV kernel, and the smallest split of
// the persistent decode kernel (whose split length the step plan chooses per
// step and stores in header[5]).  Workspaces are sized for this split.
constexpr int kSplitKeys = 512;

// Query rows per prefill unit (two 128-row tiles).
constexpr int kPrefillPairRows = 256;
// Partial-result slots for prefill units cut into KV segments: a step is
// segmented only if its segments fit.
constexpr int kPrefillSegSlots = 1024;
// Arrival tickets per partial slot: one per (query tile, softmax warp).
constexpr int kSegTicketsPerSlot = 8;

// The step's work lists, built on the GPU from the packed metadata by
// launch_plan and consumed by the persistent decode and prefill kernels, which
// claim items through the counters in `header`.  All pointers are into the
// caller's workspace.
struct StepPlan {
  int32_t* header;        // [0] decode items, [1] prefill units, [2] decode claims, [3] prefill claims,
                          // [4] call tag, [5] keys per decode split, [6] num_seqs, [7] num_tokens,
                          // [8] prefill CTAs that work (the rest leave their SMs to decode),
                          // [9] KV tiles per prefill segment (0: units are not segmented),
                          // [10] / [11] prefill / decode CTAs done claiming (the last resets
                          // its claim counter, so every launch over a plan starts at zero)
  int2* dec_items;        // (sequence, split) of every q_len == 1 row, longest first
  int2* dec_scratch;      // the decode items before sorting
  int2* pre_seqs;         // (sequence, query pairs) of every q_len > 1 chunk, costliest chunk first
  int2* pre_scratch;      // the same records before sorting
  int4* pre_units;        // prefill entries (sequence, pair | head << 16, first | end KV tile << 16,
                          // partial slot of the unit's first segment or -1), in claim order
  int32_t* pre_tickets;   // [kPrefillSegSlots][kSegTicketsPerSlot] arrival counters of segmented units
  float* pre_partials;    // [kPrefillSegSlots][A + 2][256 rows] segment results (acc, max, sum),
                          // present (else null) when num_tokens > num_seqs and
                          // max_context_len > 2048
  int32_t* tickets;       // [num_seqs][H] split arrival counters, zeroed by the plan
  float* partials;        // [num_seqs][H][max_splits][A + 2] split results (acc, max, sum)
  int32_t max_splits;
  int32_t dec_cap;        // capacity of dec_items
  int32_t pre_cap;        // capacity of pre_seqs and pre_scratch (pre_units holds pre_cap * H + kPrefillSegSlots)
  uint32_t tag;           // this call's tag: the plan writes it to header[4], the kernels check it
  int32_t dec_ctas;       // CTAs of the persistent decode grid (sets the split length)
  int32_t dec_groups;     // decode units per decode item (query-head groups)
  float dec_units_per_cta[2];    // decode units per CTA the split length aims for: [0] in a
                                 // decode-only step, [1] when prefill chunks share the step
  int32_t num_sms;        // SMs of the device (sets the prefill CTAs of a mixed step)
  int32_t kv_bytes_per_key;  // K and V bytes of one key over all key/value heads
  float dec_bytes_per_us_per_sm;  // decode K/V bytes one SM streams per microsecond
  int32_t split_sms;      // 1: a mixed step may give prefill only a share of the SMs (the
                          // decode kernel then starts behind it as a dependent launch)
};
// Decode K/V bytes one SM streams per microsecond when each unit serves
// `group_heads` query heads (measured on GB300: ~90 GB/s for one head, where
// memory binds; ~32 GB/s for four, where the arithmetic does).
float decode_rate_per_sm(int group_heads);
// Fills the decode fields of a step plan (grid size, groups, units per CTA,
// bytes per key and the decode rate of the SM-share model) for these args.
void set_decode_plan(const AttnArgs& a, StepPlan* plan);

// Workspace of a bf16 step (plan + split scratch) and its carving.
size_t step_workspace_bytes(int32_t num_seqs, int32_t num_tokens, int32_t num_heads, int32_t head_dim,
                            int32_t max_context_len);
cb_status step_plan_layout(void* workspace, size_t workspace_bytes, int32_t num_seqs, int32_t num_tokens,
                           int32_t num_heads, int32_t head_dim, int32_t max_context_len, StepPlan* plan);

// One CTA: validates every sequence's metadata (flagging bad rows in the
// error word and leaving them out), fills the work lists and clears the
// claim counters and the split tickets.  Dependent kernels launched with
// launch_after_plan may start while it runs and wait for it on the device.
cb_status launch_plan(const AttnArgs& a, const StepPlan& plan, cudaStream_t stream);

// CTAs of the persistent decode grid on the current device (0 on error), and
// the query heads each of its units covers.
int decode_persistent_ctas(const AttnArgs& a);
int decode_group_heads(const AttnArgs& a);
// Decode K/V bytes one SM streams per microsecond on the path `a` takes.
float decode_rate_for(const AttnArgs& a);

// Persistent decode over the plan's decode items (bf16, head_dim 128, block
// size a multiple of 16).  `after_previous`: a programmatic dependent launch
// behind the kernel launched just before on the same stream; `wait_previous`:
// the kernel waits for that one to finish before reading the plan (false
// when it is the prefill kernel, which releases its dependents only after
// the plan it follows is complete).
cb_status launch_decode_persistent(const AttnArgs& a, const StepPlan& plan, bool after_previous,
                                   bool wait_previous, cudaStream_t stream);

// Split-KV attention on CUDA cores.  Decode mode: one query row per sequence
// with q_len == 1 (other sequences are left to the prefill kernel).  Row mode:
// every packed row of every sequence.
size_t split_kv_workspace_bytes(bool row_mode, int32_t num_seqs, int32_t num_tokens,
                                int32_t num_heads, int32_t head_dim, int32_t max_context_len);
cb_status launch_split_kv(const AttnArgs& a, bool row_mode, void* workspace,
                          size_t workspace_bytes, cudaStream_t stream);

// Decode rows with grouped key/value heads (4 < G <= 32 query heads per
// key/value head, bf16, head_dim 128, power-of-two block size in [16, 128])
// on tcgen05 tensor cores: persistent, one CTA per SM, one unit per
// (decode item, key/value head).  decode_tc_ctas sets the kernel's shared
// memory limit once per device and returns its grid size (0 on error).
bool decode_tc_applies(const AttnArgs& a);
float decode_tc_rate_per_sm(int group_heads);
int decode_tc_ctas();
cb_status launch_decode_tc(const AttnArgs& a, const StepPlan& plan, bool after_previous, bool wait_previous,
                           cudaStream_t stream);

// Prefill chunks (q_len > 1) on tcgen05 tensor cores, bf16, head_dim 128:
// persistent CTAs over the plan's prefill items.
cb_status launch_prefill_tc(const AttnArgs& a, const StepPlan& plan, bool after_plan, cudaStream_t stream);

}  // namespace cb
