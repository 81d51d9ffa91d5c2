// cb_ragged_attention: argument checks and routing of one packed step.
//
// Hugging Face blog "Continuous batching from first principles", section
// "Continuous batching": decode tokens and prefill chunks share one step;
// page "continuous-batching", section "Inside the kernel": the attention
// kernel splits the work by request.  Here a request's rows go to one of two
// kernels by shape: q_len == 1 (decode) to split-KV on CUDA cores, which is
// bound by HBM; q_len > 1 (a prefill chunk) to tcgen05 tensor cores, which is
// a dense contraction.  A one-CTA plan kernel first lists the step's work
// units on the GPU; both attention kernels are persistent grids that claim
// those units, so the launch shape does not depend on the batch.  In a mixed
// step the prefill kernel keeps the share of SMs the plan gives it and the
// decode kernel takes the rest, side by side.  fp32 caches take the CUDA-core
// kernel for every row.
#include <cmath>
#include <mutex>
#include <unordered_map>

#include "kernels.h"
#include "runtime.h"

namespace {

bool is_pow2(int32_t x) { return x > 0 && (x & (x - 1)) == 0; }

cb_status check_cache(const cb_kv_cache* c, const char* who) {
  if (!c) return cb::fail(CB_ERR_INVALID, "%s: null cache", who);
  if (c->num_blocks < 1 || c->block_size < 1 || c->num_heads < 1 || c->head_dim < 1)
    return cb::fail(CB_ERR_INVALID, "%s: cache dimensions must be >= 1", who);
  if (c->dtype == CB_DTYPE_BF16) {
    if (c->head_dim != 128)
      return cb::fail(CB_ERR_UNSUPPORTED, "%s: bf16 needs head_dim 128", who);
    if (!is_pow2(c->block_size) || c->block_size < 8 || c->block_size > 128)
      return cb::fail(CB_ERR_UNSUPPORTED, "%s: bf16 needs block_size in {8,16,32,64,128}", who);
  } else if (c->dtype == CB_DTYPE_F32) {
    if (c->head_dim != 64 && c->head_dim != 128)
      return cb::fail(CB_ERR_UNSUPPORTED, "%s: f32 needs head_dim 64 or 128", who);
  } else {
    return cb::fail(CB_ERR_UNSUPPORTED, "%s: unknown dtype", who);
  }
  return CB_OK;
}

}  // namespace

extern "C" size_t cb_attention_workspace_size(const cb_kv_cache* cache, int32_t num_seqs,
                                              int32_t num_tokens, int32_t max_context_len) {
  if (!cache || num_seqs < 0 || num_tokens < 0 || max_context_len < 0) return 0;
  const bool row_mode = cache->dtype == CB_DTYPE_F32;
  return cb::split_kv_workspace_bytes(row_mode, num_seqs, num_tokens, cache->num_heads,
                                      cache->head_dim, max_context_len);
}

namespace {

// Host-side checks shared by every attention entry point; fills `a`.
cb_status prepare(const char* who, const void* q, const cb_kv_cache* cache, const int32_t* cu_seqlens_q,
                  const int32_t* context_lens, const int32_t* block_tables, int32_t num_seqs, int32_t num_tokens,
                  int32_t max_blocks_per_seq, int32_t max_q_len, int32_t max_context_len, float scale, void* out,
                  const int32_t* dims, bool plan_only, cb::AttnArgs& a, int32_t num_q_heads = 0) {
  cb_status st = check_cache(cache, who);
  if (st != CB_OK) return st;
  if (num_q_heads == 0) num_q_heads = cache->num_heads;
  if (num_q_heads < 1 || num_q_heads % cache->num_heads != 0)
    return cb::fail(CB_ERR_INVALID, "%s: num_q_heads must be a positive multiple of the cache's heads", who);
  if (num_q_heads != cache->num_heads && (cache->dtype != CB_DTYPE_BF16 || cache->block_size % 16 != 0))
    return cb::fail(CB_ERR_UNSUPPORTED, "%s: grouped KV heads need bf16 and a block size multiple of 16", who);
  if (num_seqs < 0 || num_tokens < 0 || max_blocks_per_seq < 0 || max_q_len < 0 || max_context_len < 0)
    return cb::fail(CB_ERR_INVALID, "%s: negative size", who);
  if (num_seqs == 0 || num_tokens == 0) {
    if ((num_seqs == 0) != (num_tokens == 0))
      return cb::fail(CB_ERR_INVALID, "%s: num_seqs and num_tokens must both be zero or both positive", who);
    return CB_OK;
  }
  if (!dims && num_tokens < num_seqs) return cb::fail(CB_ERR_INVALID, "%s: fewer tokens than sequences", who);
  if (max_q_len < 1 || max_q_len > num_tokens || max_context_len < max_q_len)
    return cb::fail(CB_ERR_INVALID, "%s: need 1 <= max_q_len <= num_tokens and max_q_len <= max_context_len", who);
  if (int64_t(max_blocks_per_seq) * cache->block_size < max_context_len)
    return cb::fail(CB_ERR_INVALID, "%s: max_blocks_per_seq * block_size < max_context_len", who);
  if (!cu_seqlens_q || !context_lens) return cb::fail(CB_ERR_INVALID, "%s: null pointer", who);
  if (!plan_only) {
    if (!(scale > 0.f) || !std::isfinite(scale))
      return cb::fail(CB_ERR_INVALID, "%s: scale must be finite and > 0", who);
    if (!q || !block_tables || !out || !cache->k || !cache->v) return cb::fail(CB_ERR_INVALID, "%s: null pointer", who);
    const uintptr_t align = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out) |
                            reinterpret_cast<uintptr_t>(cache->k) | reinterpret_cast<uintptr_t>(cache->v);
    if (align % 16 != 0) return cb::fail(CB_ERR_INVALID, "%s: q, out and the pools must be 16-byte aligned", who);
  }
  unsigned* err = cb::device_error_word();
  if (!err) return CB_ERR_CUDA;
  a.q = q;
  a.out = out;
  a.k_pool = cache->k;
  a.v_pool = cache->v;
  a.cu_seqlens_q = cu_seqlens_q;
  a.context_lens = context_lens;
  a.block_tables = block_tables;
  a.num_seqs = num_seqs;
  a.num_tokens = num_tokens;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.num_blocks = cache->num_blocks;
  a.block_size = cache->block_size;
  a.num_heads = num_q_heads;
  a.num_kv_heads = cache->num_heads;
  a.head_dim = cache->head_dim;
  a.max_q_len = max_q_len;
  a.max_context_len = max_context_len;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.dtype = cache->dtype;
  a.err = err;
  a.dims = dims;
  return CB_OK;
}

// A mixed step on one stream: the prefill kernel, then the decode kernel as a
// programmatic dependent launch.  Each prefill CTA releases its dependents
// once it has read the plan, and those beyond the plan's SM share exit at
// once.  So the decode grid starts on every SM the prefill does not keep,
// and the two run side by side (a prefill CTA's shared memory leaves no room
// for a decode CTA on its SM).  Planned steps, made to be captured in CUDA
// graphs, keep prefill on every SM: a captured step was measured to run the
// two kernels one after the other, so a share would only slow the prefill.
cb_status run_both(const cb::AttnArgs& a, const cb::StepPlan& plan, bool after_plan, cudaStream_t main) {
  cb_status st = cb::launch_prefill_tc(a, plan, after_plan, main);
  if (st != CB_OK) return st;
  return cb::launch_decode_persistent(a, plan, true, false, main);
}

// Plans built by cb_plan_step, by workspace: what the planned attention calls
// must match.
struct PlanRecord {
  cb::StepPlan plan;
  const int32_t *cu, *ctx, *dims;
  int32_t num_seqs, num_tokens, max_blocks_per_seq, max_q_len, max_context_len;
  int32_t num_q_heads, num_heads, head_dim, block_size, num_blocks;
  size_t workspace_bytes;
};
std::mutex g_plans_mutex;
std::unordered_map<const void*, PlanRecord> g_plans;

}  // namespace

namespace {

cb_status attention(const char* who, const void* q, int32_t num_q_heads, const cb_kv_cache* cache,
                    const int32_t* cu_seqlens_q, const int32_t* context_lens, const int32_t* block_tables,
                    int32_t num_seqs, int32_t num_tokens, int32_t max_blocks_per_seq, int32_t max_q_len,
                    int32_t max_context_len, float scale, void* out, void* workspace, size_t workspace_bytes,
                    void* stream, const int32_t* pad_lens = nullptr) {
  cb::AttnArgs a;
  cb_status st = prepare(who, q, cache, cu_seqlens_q, context_lens, block_tables, num_seqs, num_tokens,
                         max_blocks_per_seq, max_q_len, max_context_len, scale, out, nullptr, false, a, num_q_heads);
  if (st != CB_OK || num_seqs == 0) return st;
  a.pad_lens = pad_lens;
  cudaStream_t main = static_cast<cudaStream_t>(stream);
  if (cache->dtype == CB_DTYPE_F32) {
    if (pad_lens) return cb::fail(CB_ERR_UNSUPPORTED, "%s: padded batches need a bf16 cache", who);
    return cb::launch_split_kv(a, true, workspace, workspace_bytes, main);
  }

  // bf16: the step plan first, then the persistent kernels over its work lists
  cb::StepPlan plan;
  st = cb::step_plan_layout(workspace, workspace_bytes, num_seqs, num_tokens, a.num_heads, cache->head_dim,
                            max_context_len, &plan);
  if (st != CB_OK) return st;
  cb::set_decode_plan(a, &plan);
  plan.split_sms = 1;
  st = cb::launch_plan(a, plan, main);
  if (st != CB_OK) return st;
  if (max_q_len == 1) return cb::launch_decode_persistent(a, plan, true, true, main);
  if (max_q_len == num_tokens && num_seqs == 1) return cb::launch_prefill_tc(a, plan, true, main);
  return run_both(a, plan, true, main);
}

}  // namespace

extern "C" cb_status cb_ragged_attention(const void* q, const cb_kv_cache* cache,
                                         const int32_t* cu_seqlens_q, const int32_t* context_lens,
                                         const int32_t* block_tables, int32_t num_seqs,
                                         int32_t num_tokens, int32_t max_blocks_per_seq,
                                         int32_t max_q_len, int32_t max_context_len, float scale,
                                         void* out, void* workspace, size_t workspace_bytes,
                                         void* stream) {
  return attention("cb_ragged_attention", q, 0, cache, cu_seqlens_q, context_lens, block_tables, num_seqs,
                   num_tokens, max_blocks_per_seq, max_q_len, max_context_len, scale, out, workspace,
                   workspace_bytes, stream);
}

extern "C" cb_status cb_padded_attention(const void* q, const cb_kv_cache* cache,
                                         const int32_t* cu_seqlens_q, const int32_t* context_lens,
                                         const int32_t* block_tables, const int32_t* pad_lens,
                                         int32_t num_seqs, int32_t num_tokens, int32_t max_blocks_per_seq,
                                         int32_t max_q_len, int32_t max_context_len, float scale,
                                         void* out, void* workspace, size_t workspace_bytes,
                                         void* stream) {
  if (!pad_lens && num_seqs > 0) return cb::fail(CB_ERR_INVALID, "cb_padded_attention: null pad_lens");
  return attention("cb_padded_attention", q, 0, cache, cu_seqlens_q, context_lens, block_tables, num_seqs,
                   num_tokens, max_blocks_per_seq, max_q_len, max_context_len, scale, out, workspace,
                   workspace_bytes, stream, pad_lens);
}

extern "C" size_t cb_attention_workspace_size_gqa(const cb_kv_cache* cache, int32_t num_q_heads,
                                                  int32_t num_seqs, int32_t num_tokens,
                                                  int32_t max_context_len) {
  if (!cache || num_q_heads < 1 || num_seqs < 0 || num_tokens < 0 || max_context_len < 0) return 0;
  const bool row_mode = cache->dtype == CB_DTYPE_F32;
  return cb::split_kv_workspace_bytes(row_mode, num_seqs, num_tokens, num_q_heads, cache->head_dim,
                                      max_context_len);
}

extern "C" cb_status cb_ragged_attention_gqa(const void* q, int32_t num_q_heads, const cb_kv_cache* cache,
                                             const int32_t* cu_seqlens_q, const int32_t* context_lens,
                                             const int32_t* block_tables, int32_t num_seqs,
                                             int32_t num_tokens, int32_t max_blocks_per_seq,
                                             int32_t max_q_len, int32_t max_context_len, float scale,
                                             void* out, void* workspace, size_t workspace_bytes,
                                             void* stream) {
  if (num_q_heads < 1) return cb::fail(CB_ERR_INVALID, "cb_ragged_attention_gqa: num_q_heads < 1");
  return attention("cb_ragged_attention_gqa", q, num_q_heads, cache, cu_seqlens_q, context_lens, block_tables,
                   num_seqs, num_tokens, max_blocks_per_seq, max_q_len, max_context_len, scale, out, workspace,
                   workspace_bytes, stream);
}

namespace {

// cb_plan_step for num_q_heads query heads (a multiple of the cache's heads).
cb_status plan_step(const char* who, const cb_kv_cache* cache, int32_t num_q_heads, const int32_t* cu_seqlens_q,
                    const int32_t* context_lens, const int32_t* dims, int32_t num_seqs, int32_t num_tokens,
                    int32_t max_blocks_per_seq, int32_t max_q_len, int32_t max_context_len, void* workspace,
                    size_t workspace_bytes, void* stream) {
  if (!cache) return cb::fail(CB_ERR_INVALID, "%s: null cache", who);
  if (cache->dtype != CB_DTYPE_BF16 || cache->block_size % 16 != 0)
    return cb::fail(CB_ERR_UNSUPPORTED, "%s: planned steps need bf16 and a block size multiple of 16", who);
  // the plan reads only the metadata (q, out, block tables and pools are not needed)
  cb::AttnArgs a;
  cb_status st = prepare(who, nullptr, cache, cu_seqlens_q, context_lens, nullptr, num_seqs, num_tokens,
                         max_blocks_per_seq, max_q_len, max_context_len, 1.0f, nullptr, dims, true, a,
                         num_q_heads);
  if (st != CB_OK) return st;
  if (num_seqs == 0) return CB_OK;
  PlanRecord rec;
  st = cb::step_plan_layout(workspace, workspace_bytes, num_seqs, num_tokens, a.num_heads, cache->head_dim,
                            max_context_len, &rec.plan);
  if (st != CB_OK) return st;
  cb::set_decode_plan(a, &rec.plan);
  st = cb::launch_plan(a, rec.plan, static_cast<cudaStream_t>(stream));
  if (st != CB_OK) return st;
  rec.cu = cu_seqlens_q;
  rec.ctx = context_lens;
  rec.dims = dims;
  rec.num_seqs = num_seqs;
  rec.num_tokens = num_tokens;
  rec.max_blocks_per_seq = max_blocks_per_seq;
  rec.max_q_len = max_q_len;
  rec.max_context_len = max_context_len;
  rec.num_q_heads = a.num_heads;
  rec.num_heads = cache->num_heads;
  rec.head_dim = cache->head_dim;
  rec.block_size = cache->block_size;
  rec.num_blocks = cache->num_blocks;
  rec.workspace_bytes = workspace_bytes;
  std::lock_guard<std::mutex> lock(g_plans_mutex);
  g_plans[workspace] = rec;
  return CB_OK;
}

// cb_ragged_attention_planned for num_q_heads query heads.
cb_status attention_planned(const char* who, const void* q, int32_t num_q_heads, const cb_kv_cache* cache,
                            const int32_t* cu_seqlens_q, const int32_t* context_lens,
                            const int32_t* block_tables, const int32_t* dims, int32_t num_seqs,
                            int32_t num_tokens, int32_t max_blocks_per_seq, int32_t max_q_len,
                            int32_t max_context_len, float scale, void* out, void* workspace,
                            size_t workspace_bytes, void* stream) {
  cb::AttnArgs a;
  cb_status st = prepare(who, q, cache, cu_seqlens_q, context_lens, block_tables, num_seqs, num_tokens,
                         max_blocks_per_seq, max_q_len, max_context_len, scale, out, dims, false, a,
                         num_q_heads);
  if (st != CB_OK || num_seqs == 0) return st;
  PlanRecord rec;
  {
    std::lock_guard<std::mutex> lock(g_plans_mutex);
    auto it = g_plans.find(workspace);
    if (it == g_plans.end()) return cb::fail(CB_ERR_INVALID, "%s: no cb_plan_step was made in this workspace", who);
    rec = it->second;
  }
  if (rec.cu != cu_seqlens_q || rec.ctx != context_lens || rec.dims != dims || rec.num_seqs != num_seqs ||
      rec.num_tokens != num_tokens || rec.max_blocks_per_seq != max_blocks_per_seq || rec.max_q_len != max_q_len ||
      rec.max_context_len != max_context_len || rec.num_q_heads != a.num_heads ||
      rec.num_heads != cache->num_heads ||
      rec.head_dim != cache->head_dim || rec.block_size != cache->block_size ||
      rec.num_blocks != cache->num_blocks || rec.workspace_bytes != workspace_bytes)
    return cb::fail(CB_ERR_INVALID, "%s: the workspace's plan was made for other metadata, sizes or cache shape",
                    who);
  cudaStream_t main = static_cast<cudaStream_t>(stream);
  // The claim counters are back at zero: the plan zeroes them and every
  // persistent grid's last CTA resets its own.  The prefill kernel goes out
  // as a programmatic dependent of whatever kernel precedes it (the layer's
  // append): it waits for that grid on the device before reading anything,
  // so only its launch overlaps.
  return run_both(a, rec.plan, true, main);
}

}  // namespace

extern "C" cb_status cb_plan_step(const cb_kv_cache* cache, const int32_t* cu_seqlens_q,
                                  const int32_t* context_lens, const int32_t* dims, int32_t num_seqs,
                                  int32_t num_tokens, int32_t max_blocks_per_seq, int32_t max_q_len,
                                  int32_t max_context_len, void* workspace, size_t workspace_bytes,
                                  void* stream) {
  return plan_step("cb_plan_step", cache, 0, cu_seqlens_q, context_lens, dims, num_seqs, num_tokens,
                   max_blocks_per_seq, max_q_len, max_context_len, workspace, workspace_bytes, stream);
}

extern "C" cb_status cb_plan_step_gqa(const cb_kv_cache* cache, int32_t num_q_heads,
                                      const int32_t* cu_seqlens_q, const int32_t* context_lens,
                                      const int32_t* dims, int32_t num_seqs, int32_t num_tokens,
                                      int32_t max_blocks_per_seq, int32_t max_q_len, int32_t max_context_len,
                                      void* workspace, size_t workspace_bytes, void* stream) {
  if (num_q_heads < 1) return cb::fail(CB_ERR_INVALID, "cb_plan_step_gqa: num_q_heads < 1");
  return plan_step("cb_plan_step_gqa", cache, num_q_heads, cu_seqlens_q, context_lens, dims, num_seqs,
                   num_tokens, max_blocks_per_seq, max_q_len, max_context_len, workspace, workspace_bytes,
                   stream);
}

extern "C" cb_status cb_ragged_attention_planned(const void* q, const cb_kv_cache* cache,
                                                 const int32_t* cu_seqlens_q, const int32_t* context_lens,
                                                 const int32_t* block_tables, const int32_t* dims,
                                                 int32_t num_seqs, int32_t num_tokens,
                                                 int32_t max_blocks_per_seq, int32_t max_q_len,
                                                 int32_t max_context_len, float scale, void* out,
                                                 void* workspace, size_t workspace_bytes, void* stream) {
  return attention_planned("cb_ragged_attention_planned", q, 0, cache, cu_seqlens_q, context_lens, block_tables,
                           dims, num_seqs, num_tokens, max_blocks_per_seq, max_q_len, max_context_len, scale,
                           out, workspace, workspace_bytes, stream);
}

extern "C" cb_status cb_ragged_attention_planned_gqa(const void* q, int32_t num_q_heads,
                                                     const cb_kv_cache* cache, const int32_t* cu_seqlens_q,
                                                     const int32_t* context_lens, const int32_t* block_tables,
                                                     const int32_t* dims, int32_t num_seqs, int32_t num_tokens,
                                                     int32_t max_blocks_per_seq, int32_t max_q_len,
                                                     int32_t max_context_len, float scale, void* out,
                                                     void* workspace, size_t workspace_bytes, void* stream) {
  if (num_q_heads < 1) return cb::fail(CB_ERR_INVALID, "cb_ragged_attention_planned_gqa: num_q_heads < 1");
  return attention_planned("cb_ragged_attention_planned_gqa", q, num_q_heads, cache, cu_seqlens_q, context_lens,
                           block_tables, dims, num_seqs, num_tokens, max_blocks_per_seq, max_q_len,
                           max_context_len, scale, out, workspace, workspace_bytes, stream);
}
