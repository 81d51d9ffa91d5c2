// cb_decode_attention_noalloc: the split-KV decode kernel with its scratch
// (split tickets and fp32 partials) in a fixed array that the library reserves
// in device memory, so the call itself allocates nothing.
//
// For callers that cannot allocate device memory and cannot lend a workspace:
// e.g. an op running inside a host framework whose caching allocator, or a KV
// pool sized to fill the GPU, already owns all device memory, behind a plugin
// interface that passes only the op's inputs and outputs.
#include <mutex>

#include "kernels.h"
#include "runtime.h"

namespace {

// Reserved on every device that loads the library, for the life of the process.
static __device__ __align__(256) unsigned char g_decode_scratch[CB_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  The host-side
// symbol is only a stand-in; the address comes from cudaGetSymbolAddress with
// the device current, once per device.
cb_status scratch_for_current_device(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cb::cuda_fail(e, "cb_decode_attention_noalloc: cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices)
    return cb::fail(CB_ERR_UNSUPPORTED, "cb_decode_attention_noalloc: device index %d", dev);
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess || !p)
      return cb::cuda_fail(e, "cb_decode_attention_noalloc: cudaGetSymbolAddress(scratch)");
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return CB_OK;
}

}  // namespace

extern "C" cb_status cb_decode_attention_noalloc(const void* q, const cb_kv_cache* cache,
                                                 const int32_t* cu_seqlens_q,
                                                 const int32_t* context_lens,
                                                 const int32_t* block_tables, int32_t num_seqs,
                                                 int32_t num_tokens, int32_t max_blocks_per_seq,
                                                 int32_t max_context_len, float scale, void* out,
                                                 void* stream) {
  const char* who = "cb_decode_attention_noalloc";
  if (!cache) return cb::fail(CB_ERR_INVALID, "%s: null cache", who);
  if (cache->num_blocks < 1 || cache->block_size < 1 || cache->num_heads < 1)
    return cb::fail(CB_ERR_INVALID, "%s: cache dimensions must be >= 1", who);
  const bool bf16 = cache->dtype == CB_DTYPE_BF16;
  if (!bf16 && cache->dtype != CB_DTYPE_F32) return cb::fail(CB_ERR_UNSUPPORTED, "%s: unknown dtype", who);
  if ((bf16 && cache->head_dim != 128) || (!bf16 && cache->head_dim != 64 && cache->head_dim != 128))
    return cb::fail(CB_ERR_UNSUPPORTED, "%s: head_dim must be 128 (bf16) or 64/128 (f32)", who);
  if (num_seqs < 0 || max_blocks_per_seq < 0 || max_context_len < 0)
    return cb::fail(CB_ERR_INVALID, "%s: negative size", who);
  if (num_tokens != num_seqs)
    return cb::fail(CB_ERR_INVALID, "%s: decode only: every sequence must have exactly one query token", who);
  if (num_seqs == 0) return CB_OK;
  if (max_context_len < 1 || int64_t(max_blocks_per_seq) * cache->block_size < max_context_len)
    return cb::fail(CB_ERR_INVALID, "%s: need max_context_len >= 1 and max_blocks_per_seq * block_size >= max_context_len", who);
  if (!(scale > 0.f) || scale == INFINITY) return cb::fail(CB_ERR_INVALID, "%s: scale must be finite and > 0", who);
  const size_t need = cb::split_kv_workspace_bytes(false, num_seqs, num_tokens, cache->num_heads,
                                                   cache->head_dim, max_context_len);
  if (need > size_t(CB_NOALLOC_SCRATCH_BYTES))
    return cb::fail(CB_ERR_INVALID,
                    "%s: this step needs %zu bytes of scratch but the static scratch holds %zu; use "
                    "cb_ragged_attention with a caller workspace",
                    who, need, size_t(CB_NOALLOC_SCRATCH_BYTES));
  if (!q || !cu_seqlens_q || !context_lens || !block_tables || !out || !cache->k || !cache->v)
    return cb::fail(CB_ERR_INVALID, "%s: null pointer", who);
  const uintptr_t align = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out) |
                          reinterpret_cast<uintptr_t>(cache->k) | reinterpret_cast<uintptr_t>(cache->v);
  if (align % 16 != 0) return cb::fail(CB_ERR_INVALID, "%s: q, out and the pools must be 16-byte aligned", who);

  void* scratch = nullptr;
  cb_status st = scratch_for_current_device(&scratch);
  if (st != CB_OK) return st;
  unsigned* err = cb::device_error_word();
  if (!err) return CB_ERR_CUDA;
  cb::AttnArgs a;
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
  a.num_heads = cache->num_heads;
  a.num_kv_heads = cache->num_heads;
  a.head_dim = cache->head_dim;
  a.max_q_len = 1;
  a.max_context_len = max_context_len;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.dtype = cache->dtype;
  a.err = err;
  // The split tickets and claim counters must start at zero, whatever the
  // previous call left in the array: the step-plan kernel that launch_split_kv
  // runs first zeroes them, on the same stream, before the decode kernel
  // reads them.
  return cb::launch_split_kv(a, false, scratch, size_t(CB_NOALLOC_SCRATCH_BYTES),
                             static_cast<cudaStream_t>(stream));
}
