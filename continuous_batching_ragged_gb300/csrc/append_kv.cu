// K1: append this step's keys and values to the block-paged cache.
//
// Page "continuous-batching" (zhangchitc.github.io), section "Inside the
// kernel": the new keys and values are written into the KV cache, each into
// its own request's entry, before attention reads the cache back.
//
// A pure copy, HBM-bound: each thread moves one 16-byte chunk of one (token,
// head) row of K or V.  Source reads are fully contiguous; a (token, head) row
// of head_dim * elem bytes lands contiguously at pool[block][h][offset][:].
#include <algorithm>

#include "device_common.cuh"
#include "runtime.h"

namespace {

__global__ void __launch_bounds__(256) append_kv_kernel(
    const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
    const int64_t* __restrict__ slot_mapping, uint4* __restrict__ k_pool,
    uint4* __restrict__ v_pool, int64_t chunks_per_tensor, int32_t heads_x_chunks,
    int32_t chunks_per_row, int32_t num_heads, int32_t block_size, int64_t num_slots,
    const int32_t* __restrict__ dims, unsigned* err) {
  // dims: the step's token count comes from device memory (dims[1], at most
  // the chunks_per_tensor the launch was sized for); the grid strides over it
  int64_t per_tensor = chunks_per_tensor;
  if (dims) {
    const int32_t t = dims[1];
    const int64_t n = int64_t(t) * heads_x_chunks;
    if (t < 0 || n > chunks_per_tensor) {
      if (blockIdx.x == 0 && threadIdx.x == 0) cb::raise_error(err, cb::kErrInvalid);
      return;
    }
    per_tensor = n;
  }
  for (int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; idx < 2 * per_tensor;
       idx += int64_t(gridDim.x) * blockDim.x) {
    const bool is_v = idx >= per_tensor;
    const int64_t i = is_v ? idx - per_tensor : idx;
    const int64_t t = i / heads_x_chunks;
    const int32_t rem = int32_t(i - t * heads_x_chunks);
    const int32_t h = rem / chunks_per_row;
    const int32_t c = rem - h * chunks_per_row;
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= num_slots) {
      cb::raise_error(err, cb::kErrBounds);
      continue;
    }
    const int64_t blk = slot / block_size;
    const int64_t off = slot - blk * block_size;
    const uint4 val = is_v ? cb::ldg_stream(v_new + i) : cb::ldg_stream(k_new + i);
    uint4* pool = is_v ? v_pool : k_pool;
    pool[((blk * num_heads + h) * block_size + off) * chunks_per_row + c] = val;
  }
}

cb_status append(const void* k_new, const void* v_new, const int64_t* slot_mapping, int32_t num_tokens,
                 const int32_t* dims, const cb_kv_cache* cache, void* stream, const char* who) {
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
  const int32_t heads_x_chunks = chunks_per_row * cache->num_heads;
  const int64_t per_tensor = int64_t(num_tokens) * heads_x_chunks;
  const int64_t threads = 2 * per_tensor;
  const int block = 256;
  int64_t grid = (threads + block - 1) / block;
  // with device sizes the step may be far below the capacity: a grid of a few
  // CTAs per SM strides over whatever the step holds
  if (dims) grid = std::min<int64_t>(grid, int64_t(cb::sm_count()) * 8);
  if (grid > 0x7FFFFFFF) return cb::fail(CB_ERR_INVALID, "%s: too many tokens", who);
  append_kv_kernel<<<unsigned(grid), block, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), slot_mapping,
      static_cast<uint4*>(cache->k), static_cast<uint4*>(cache->v), per_tensor, heads_x_chunks,
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
