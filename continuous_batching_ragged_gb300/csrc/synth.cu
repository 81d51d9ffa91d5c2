// Seeded synthetic inputs in device memory (see cb_synth.h for the definition).
// Philox4x32-10: Salmon, Moraes, Dror, Shaw, SC'11.  Every operation below is
// exact integer arithmetic or one correctly rounded fp32 operation, so the
// values match an independent host implementation bit for bit.
#include <cuda_bf16.h>

#include "cb_synth.h"
#include "device_common.cuh"
#include "runtime.h"

namespace {

struct U4 {
  uint32_t x, y, z, w;
};

__device__ __forceinline__ U4 philox4x32_10(U4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = U4{hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0};
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}

__device__ __forceinline__ float irwin_hall8(U4 w) {
  const int32_t s = int32_t((w.x & 0xFFFFu) + (w.x >> 16) + (w.y & 0xFFFFu) + (w.y >> 16) +
                            (w.z & 0xFFFFu) + (w.z >> 16) + (w.w & 0xFFFFu) + (w.w >> 16));
  const int32_t s2 = 2 * s - 8 * 65535;
  return __fmul_rn(__int2float_rn(s2), __uint_as_float(0x371cc471u));  // sqrt(1.5)/131072
}

__device__ __forceinline__ float value(uint64_t seed, uint32_t tag, uint32_t seq, uint32_t pos,
                                       uint32_t elem) {
  return irwin_hall8(philox4x32_10(U4{elem, pos, seq, tag}, uint32_t(seed), uint32_t(seed >> 32)));
}

// Writes the 8 consecutive dims [d0, d0+8) of one (token, head) row.
template <typename T>
__device__ __forceinline__ void write8(T* dst, uint64_t seed, uint32_t tag, uint32_t seq,
                                       uint32_t pos, uint32_t elem0);

template <>
__device__ __forceinline__ void write8<__nv_bfloat16>(__nv_bfloat16* dst, uint64_t seed, uint32_t tag,
                                                      uint32_t seq, uint32_t pos, uint32_t elem0) {
  uint32_t packed[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float a = value(seed, tag, seq, pos, elem0 + 2 * i);
    const float b = value(seed, tag, seq, pos, elem0 + 2 * i + 1);
    __nv_bfloat162 pr = __floats2bfloat162_rn(a, b);
    packed[i] = *reinterpret_cast<uint32_t*>(&pr);
  }
  *reinterpret_cast<uint4*>(dst) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
}

template <>
__device__ __forceinline__ void write8<float>(float* dst, uint64_t seed, uint32_t tag, uint32_t seq,
                                              uint32_t pos, uint32_t elem0) {
  float v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = value(seed, tag, seq, pos, elem0 + i);
  reinterpret_cast<float4*>(dst)[0] = make_float4(v[0], v[1], v[2], v[3]);
  reinterpret_cast<float4*>(dst)[1] = make_float4(v[4], v[5], v[6], v[7]);
}

template <typename T>
__global__ void synth_tokens_kernel(T* out, uint64_t seed, uint32_t tag, const int64_t* seq_ids,
                                    const int32_t* positions, int64_t n, int32_t H, int32_t A) {
  const int64_t chunks = int64_t(H) * (A / 8);
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= n * chunks) return;
  const int64_t i = idx / chunks;
  const int32_t r = int32_t(idx - i * chunks);   // = h * (A/8) + chunk
  const uint32_t elem0 = uint32_t(r) * 8u;       // = h*A + chunk*8
  write8<T>(out + i * int64_t(H) * A + elem0, seed, tag, uint32_t(seq_ids[i]), uint32_t(positions[i]),
            elem0);
}

template <typename T>
__global__ void synth_fill_kernel(T* pool, uint64_t seed, uint32_t tag, const int64_t* seq_ids,
                                  const int32_t* prefix_lens, const int32_t* block_tables,
                                  int32_t max_blocks, int32_t num_blocks, int32_t B, int32_t H,
                                  int32_t A, unsigned* err) {
  const int s = blockIdx.z;
  const int32_t chunks = H * (A / 8);
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t pos = idx / chunks;
  if (pos >= prefix_lens[s]) return;
  const int32_t r = int32_t(idx - pos * chunks);
  const int32_t h = r / (A / 8);
  const int32_t chunk = r - h * (A / 8);
  const int64_t lb = pos / B;
  if (lb >= max_blocks) {
    cb::raise_error(err, cb::kErrBounds);
    return;
  }
  const int32_t blk = block_tables[int64_t(s) * max_blocks + lb];
  if (blk < 0 || blk >= num_blocks) {
    cb::raise_error(err, cb::kErrBounds);
    return;
  }
  T* dst = pool + ((int64_t(blk) * H + h) * B + pos % B) * A + chunk * 8;
  write8<T>(dst, seed, tag, uint32_t(seq_ids[s]), uint32_t(pos), uint32_t(r) * 8u);
}

}  // namespace

extern "C" cb_status cb_synth_tokens(void* out, cb_dtype dtype, uint64_t seed, int32_t kind,
                                     int32_t layer, const int64_t* seq_ids, const int32_t* positions,
                                     int32_t n, int32_t num_heads, int32_t head_dim, void* stream) {
  if (n < 0 || num_heads < 1 || head_dim < 8 || head_dim % 8 != 0)
    return cb::fail(CB_ERR_INVALID, "cb_synth_tokens: bad sizes");
  if (n == 0) return CB_OK;
  if (!out || !seq_ids || !positions) return cb::fail(CB_ERR_INVALID, "cb_synth_tokens: null pointer");
  const uint32_t tag = (uint32_t(kind & 0xFFFF) << 16) | uint32_t(layer & 0xFFFF);
  const int64_t threads = int64_t(n) * num_heads * (head_dim / 8);
  const unsigned grid = unsigned((threads + 255) / 256);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == CB_DTYPE_BF16)
    synth_tokens_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(static_cast<__nv_bfloat16*>(out), seed, tag,
                                                             seq_ids, positions, n, num_heads, head_dim);
  else if (dtype == CB_DTYPE_F32)
    synth_tokens_kernel<float><<<grid, 256, 0, st>>>(static_cast<float*>(out), seed, tag, seq_ids,
                                                     positions, n, num_heads, head_dim);
  else
    return cb::fail(CB_ERR_UNSUPPORTED, "cb_synth_tokens: unknown dtype");
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? CB_OK : cb::cuda_fail(e, "cb_synth_tokens: launch");
}

extern "C" cb_status cb_synth_fill_cache(void* pool, cb_dtype dtype, uint64_t seed, int32_t kind,
                                         int32_t layer, const int64_t* seq_ids,
                                         const int32_t* prefix_lens, const int32_t* block_tables,
                                         int32_t num_seqs, int32_t max_blocks_per_seq,
                                         int32_t num_blocks, int32_t block_size, int32_t num_heads,
                                         int32_t head_dim, int32_t max_prefix, void* stream) {
  if (num_seqs < 0 || num_seqs > 65535 || max_prefix < 0 || num_heads < 1 || head_dim < 8 ||
      head_dim % 8 != 0 || block_size < 1 || num_blocks < 1 || max_blocks_per_seq < 0)
    return cb::fail(CB_ERR_INVALID, "cb_synth_fill_cache: bad sizes");
  if (num_seqs == 0 || max_prefix == 0) return CB_OK;
  if (!pool || !seq_ids || !prefix_lens || !block_tables)
    return cb::fail(CB_ERR_INVALID, "cb_synth_fill_cache: null pointer");
  unsigned* err = cb::device_error_word();
  if (!err) return CB_ERR_CUDA;
  const uint32_t tag = (uint32_t(kind & 0xFFFF) << 16) | uint32_t(layer & 0xFFFF);
  const int64_t per_seq = int64_t(max_prefix) * num_heads * (head_dim / 8);
  dim3 grid(unsigned((per_seq + 255) / 256), 1, unsigned(num_seqs));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == CB_DTYPE_BF16)
    synth_fill_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(
        static_cast<__nv_bfloat16*>(pool), seed, tag, seq_ids, prefix_lens, block_tables,
        max_blocks_per_seq, num_blocks, block_size, num_heads, head_dim, err);
  else if (dtype == CB_DTYPE_F32)
    synth_fill_kernel<float><<<grid, 256, 0, st>>>(static_cast<float*>(pool), seed, tag, seq_ids,
                                                   prefix_lens, block_tables, max_blocks_per_seq,
                                                   num_blocks, block_size, num_heads, head_dim, err);
  else
    return cb::fail(CB_ERR_UNSUPPORTED, "cb_synth_fill_cache: unknown dtype");
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? CB_OK : cb::cuda_fail(e, "cb_synth_fill_cache: launch");
}
