/*
 * cb_synth.h -- seeded synthetic inputs generated directly in device memory.
 *
 * Not part of the attention step: tests and benchmarks use these to create
 * workloads too large to build on the host (a decode step over ~10 GB of
 * cached keys and values).  The sources describe no such generator; the values follow a
 * published counter-based generator so that a host implementation can
 * recompute any element independently:
 *
 *   value(seed, kind, layer, seq_id, position, head, dim)
 *     = IH8(Philox4x32-10(counter = (head*A + dim, position, seq_id, kind<<16 | layer),
 *                         key     = (seed mod 2^32, seed >> 32)))
 *
 * Philox4x32-10 is the generator of Salmon, Moraes, Dror and Shaw, "Parallel
 * random numbers: as easy as 1, 2, 3" (SC'11).  IH8 splits the four output
 * words into eight 16-bit uniforms u_k and returns the exact fp32 product
 * fp32(2*sum(u_k) - 8*65535) * fp32(sqrt(1.5)/131072) -- an Irwin-Hall(8)
 * approximation of N(0,1) -- rounded to nearest-even bf16 for bf16 buffers.
 * kind: 0 = query, 1 = key, 2 = value.
 */
#ifndef CB_SYNTH_H_
#define CB_SYNTH_H_

#include <stdint.h>

#include "cb.h"

#ifdef __cplusplus
extern "C" {
#endif

/* out: device [n][H][A] of dtype.  Row i holds the token (seq_ids[i],
 * positions[i]); seq_ids and positions are device arrays of n entries. */
cb_status cb_synth_tokens(void* out, cb_dtype dtype, uint64_t seed, int32_t kind, int32_t layer,
                          const int64_t* seq_ids, const int32_t* positions, int32_t n,
                          int32_t num_heads, int32_t head_dim, void* stream);

/* Write positions 0 .. prefix_lens[s]-1 of every sequence s into `pool`
 * ([num_blocks][H][block_size][A] of dtype) at the slots its block table
 * gives.  seq_ids, prefix_lens, block_tables are device arrays; max_prefix is
 * a host upper bound on prefix_lens.  Block ids outside the pool set
 * CB_ERR_BOUNDS on the device error word and are skipped. */
cb_status cb_synth_fill_cache(void* pool, cb_dtype dtype, uint64_t seed, int32_t kind,
                              int32_t layer, const int64_t* seq_ids, const int32_t* prefix_lens,
                              const int32_t* block_tables, int32_t num_seqs,
                              int32_t max_blocks_per_seq, int32_t num_blocks, int32_t block_size,
                              int32_t num_heads, int32_t head_dim, int32_t max_prefix,
                              void* stream);

#ifdef __cplusplus
}
#endif
#endif /* CB_SYNTH_H_ */
