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
  int32_t num_heads;
  int32_t head_dim;
  int32_t max_q_len;
  int32_t max_context_len;
  float scale_log2;       // softmax scale * log2(e)
  cb_dtype dtype;
  unsigned* err;
};

// Keys per split of the split-KV kernel.  The split plan of a row depends only
// on that row's own number of visible keys.
constexpr int kSplitKeys = 512;

// Split-KV attention on CUDA cores.  Decode mode: one query row per sequence
// with q_len == 1 (other sequences are left to the prefill kernel).  Row mode:
// every packed row of every sequence.
size_t split_kv_workspace_bytes(bool row_mode, int32_t num_seqs, int32_t num_tokens,
                                int32_t num_heads, int32_t head_dim, int32_t max_context_len);
cb_status launch_split_kv(const AttnArgs& a, bool row_mode, void* workspace,
                          size_t workspace_bytes, cudaStream_t stream);

// Prefill chunks (q_len > 1) on tcgen05 tensor cores, bf16, head_dim 128.
cb_status launch_prefill_tc(const AttnArgs& a, cudaStream_t stream);

}  // namespace cb
