// K1: append this step's keys and values to the block-paged cache.
//
// Page "continuous-batching" (zhangchitc.github.io), section "Inside the
// kernel": a step first stores every new key and value row under the request
// it belongs to; attention then reads the cache.
//
// A pure copy, HBM-bound.  A token's K (and V) rows are contiguous in k_new;
// a (token, head) row of head_dim * elem bytes lands contiguously at
// pool[block][h][offset][:].
#include <algorithm>

#include "device_common.cuh"
#include "runtime.h"

namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;      // 16-byte chunks in flight per thread

// One CTA per token (striding over tokens when the count comes from the
// device): its slot is read once, then the CTA copies the token's K and V
// rows, 2 * heads_x_chunks 16-byte chunks, kUnroll loads in flight per thread.
__global__ void __launch_bounds__(kThreads) append_kv_kernel(
    const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
    const int64_t* __restrict__ slot_mapping, uint4* __restrict__ k_pool,
    uint4* __restrict__ v_pool, int32_t num_tokens, int32_t heads_x_chunks,
    int32_t chunks_per_row, int32_t num_heads, int32_t block_size, int64_t num_slots,
    const int32_t* __restrict__ dims, unsigned* err) {
  int32_t T = num_tokens;
  if (dims) {                   // the step's token count, at most num_tokens (the capacity)
    const int32_t t = dims[1];
    if (t < 0 || t > num_tokens) {
      if (blockIdx.x == 0 && threadIdx.x == 0) cb::raise_error(err, cb::kErrInvalid);
      return;
    }
    T = t;
  }
  const int32_t n = 2 * heads_x_chunks;
  for (int32_t tok = blockIdx.x; tok < T; tok += gridDim.x) {
    const int64_t slot = slot_mapping[tok];
    if (slot < 0) continue;
    if (slot >= num_slots) {
      if (threadIdx.x == 0) cb::raise_error(err, cb::kErrBounds);
      continue;
    }
    const int64_t blk = slot / block_size;
    const int64_t off = slot - blk * block_size;
    const uint4* ks = k_new + int64_t(tok) * heads_x_chunks;
    const uint4* vs = v_new + int64_t(tok) * heads_x_chunks;
    const int64_t dst0 = (blk * num_heads * block_size + off) * chunks_per_row;
    const int64_t head_stride = int64_t(block_size) * chunks_per_row;
    for (int32_t i0 = threadIdx.x; i0 < n; i0 += kThreads * kUnroll) {
      uint4 val[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int32_t i = i0 + u * kThreads;
        if (i < n) val[u] = i < heads_x_chunks ? cb::ldg_stream(ks + i) : cb::ldg_stream(vs + (i - heads_x_chunks));
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int32_t i = i0 + u * kThreads;
        if (i < n) {
          const bool is_v = i >= heads_x_chunks;
          const int32_t r = is_v ? i - heads_x_chunks : i;
          const int32_t h = r / chunks_per_row;
          const int32_t c = r - h * chunks_per_row;
          (is_v ? v_pool : k_pool)[dst0 + h * head_stride + c] = val[u];
        }
      }
    }
  }
}

cb_status append(const void* k_new, const void* v_new, const int64_t* slot_mapping, int32_t num_tokens,
                 const int32_t* dims, const cb_kv_cache* cache, void* stream, const char* who) {
  cb::NvtxRange nvtx("cb.append_kv");
  if (!cache) return cb::fail(CB_ERR_INVALID, "%s: null cache", who);
  if (num_tokens < 0) return cb::fail(CB_ERR_INVALID, "%s: num_tokens < 0", who);
  if (cache->num_blocks < 1 || cache->block_size < 1 || cache->num_heads < 1 || cache->head_dim < 1)
    return cb::fail(CB_ERR_INVALID, "%s: cache dimensions must be >= 1", who);
  if (cache->dtype != CB_DTYPE_BF16 && cache->dtype != CB_DTYPE_F32)
    return cb::fail(CB_ERR_UNSUPPORTED, "%s: unknown dtype", who);
  const int elem = cache->dtype == CB_DTYPE_BF16 ? 2 : 4;
  const int64_t row_bytes = int64_t(cache->head_dim) * elem;
  if (row_bytes % 16 != 0)
    return cb::fail(CB_ERR_UNSUPPORTED, "%s: head_dim * element size must be a multiple of 16", who);
  if (num_tokens == 0) return CB_OK;
  if (!k_new || !v_new || !slot_mapping || !cache->k || !cache->v)
    return cb::fail(CB_ERR_INVALID, "%s: null pointer", who);
  const uintptr_t align = reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new) |
                          reinterpret_cast<uintptr_t>(cache->k) | reinterpret_cast<uintptr_t>(cache->v);
  if (align % 16 != 0) return cb::fail(CB_ERR_INVALID, "%s: buffers must be 16-byte aligned", who);
  unsigned* err = cb::device_error_word();
  if (!err) return CB_ERR_CUDA;

  const int32_t chunks_per_row = int32_t(row_bytes / 16);
  if (int64_t(chunks_per_row) * cache->num_heads * 2 > 0x7FFFFFFF)
    return cb::fail(CB_ERR_UNSUPPORTED, "%s: rows too wide", who);
  const int32_t heads_x_chunks = chunks_per_row * cache->num_heads;
  // one CTA per token; with device sizes the step may be far below the
  // capacity, so a few CTAs per SM stride over whatever the step holds
  int64_t grid = num_tokens;
  if (dims) grid = std::min<int64_t>(grid, int64_t(cb::sm_count()) * 2);
  append_kv_kernel<<<unsigned(grid), kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), slot_mapping,
      static_cast<uint4*>(cache->k), static_cast<uint4*>(cache->v), num_tokens, heads_x_chunks,
      chunks_per_row, cache->num_heads, cache->block_size,
      int64_t(cache->num_blocks) * cache->block_size, dims, err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cb::cuda_fail(e, "append: launch");
  return CB_OK;
}

}  // namespace

extern "C" cb_status cb_append_kv(const void* k_new, const void* v_new,
                                  const int64_t* slot_mapping, int32_t num_tokens,
                                  const cb_kv_cache* cache, void* stream) {
  return append(k_new, v_new, slot_mapping, num_tokens, nullptr, cache, stream, "cb_append_kv");
}

extern "C" cb_status cb_append_kv_dims(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                                       const int32_t* dims, int32_t max_tokens, const cb_kv_cache* cache,
                                       void* stream) {
  if (!dims) return cb::fail(CB_ERR_INVALID, "cb_append_kv_dims: null dims");
  return append(k_new, v_new, slot_mapping, max_tokens, dims, cache, stream, "cb_append_kv_dims");
}
