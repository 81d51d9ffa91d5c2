// The step plan: work lists for the persistent attention kernels, built on
// the GPU from the packed metadata.
//
// Page "continuous-batching" (zhangchitc.github.io), section "Inside the
// kernel": the loops over requests and over each request's cache become the
// kernel's parallel units.  Here the units are listed explicitly, once per
// step, so the attention kernels can run a fixed grid (one or two CTAs per SM)
// that claims units until the lists run out: no CTA is launched for a unit
// that does not exist (a split past a short context, a prefill tile of a
// decode row), and the launch shape no longer depends on the batch, which is
// what lets a whole step be captured once in a CUDA graph.
//   * decode items: (sequence, split) for every q_len == 1 row, one per
//     split of its context, sorted by length (longest first, so that greedy
//     claiming ends on short units); the split length is chosen per step;
//   * prefill units: (sequence, pair of 128-row query tiles, head) for every
//     q_len > 1 chunk; chunks by total cost (KV tiles x query tiles,
//     costliest first), then head by head, so the pairs of one (sequence,
//     head) share its K/V tiles in L2.
// A decode item stands for num_heads units, one per head.
#include <atomic>

#include "device_common.cuh"
#include "kernels.h"
#include "runtime.h"

namespace cb {
namespace {

constexpr int kPlanThreads = 256;
constexpr int kCostBuckets = 4096;     // costs at or above the last bucket share it
constexpr int kRowCache = 2048;        // rows whose (q_len, ctx) stay in shared memory after pass 1
// Cost model of a mixed step's SM split, fitted on GB300 to the long-prompt
// chunk and to %globaltimer stamps of the mixed step's two kernels running
// side by side, then retuned by timing the mixed step over the per-tile cost
// (0.9 / 1.1 / 1.3 / 1.5 us): a prefill unit costs about 2.75 us plus 1.3 us
// per (KV tile x query tile) on one SM, the rate of a prefill SM while decode
// shares the GPU's memory system; decode streams K/V at about 6.5 TB/s overall, and at
// most at the per-SM rate the host passes (lower when a unit serves several
// query heads: then the decode kernel is bound by its arithmetic, not by
// memory).  A split is taken only if it beats the two kernels one after the
// other (prefill on every SM, then decode) by kSplitGain.
constexpr float kPrefillUsPerUnit = 2.75f;
constexpr float kPrefillUsPerCost = 1.3f;
constexpr float kDecodeBytesPerUs = 6.5e6f;
constexpr float kSplitGain = 0.9f;
// Prefill KV segments: a query pair's keys are cut into segments of L KV
// tiles when some pair is long next to the work every SM gets (the step's
// prefill and decode estimates over all SMs), which otherwise leaves a tail
// of idle SMs: the last 2048-token chunk of a 32768-token prompt is 256 units
// of ~250 tiles for 152 SMs.  L is 1/kSegPerShare of an SM's share, at least
// kSegMinTiles.  The choice depends on the step and the SM count only, not on
// the SM share a mixed step gives prefill, so a step's bits never depend on it.
constexpr int kSegPerShare = 4;
constexpr int kSegMinTiles = 16;

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// Segment partials exist only where a step could use them: a prefill chunk
// (T > S) with a context longer than the shortest segment.
bool has_seg_partials(size_t S, size_t T, int32_t max_context_len) {
  return T > S && max_context_len > kSegMinTiles * 128;
}

__device__ __forceinline__ void launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Exclusive block-wide scan of 64-bit values (two 32-bit counters packed,
// which add without carries between them).  Returns this thread's prefix;
// `total` receives the block sum.  Contains __syncthreads.
__device__ uint64_t block_excl_scan(uint64_t v, uint64_t* warp_sums, uint64_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint64_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    uint64_t w = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint64_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < nw) warp_sums[lane] = w;     // inclusive warp prefixes
  }
  __syncthreads();
  total = warp_sums[(blockDim.x >> 5) - 1];
  const uint64_t before = warp == 0 ? 0 : warp_sums[warp - 1];
  const uint64_t r = before + x - v;
  __syncthreads();                          // warp_sums is reused by the next call
  return r;
}

// Prefill work of query pair qp of a chunk: KV tiles the pair streams times
// the query tiles it holds.
__device__ __forceinline__ int pair_cost(int q_len, int ctx, int qp) {
  const int row0 = qp * kPrefillPairRows;
  const int nq = row0 + kPrefillPairRows / 2 < q_len ? 2 : 1;
  const int kv_end = min(ctx - q_len + row0 + nq * (kPrefillPairRows / 2), ctx);
  return ((kv_end + 127) / 128) * nq;
}

// KV tiles that query pair qp of a chunk streams.
__device__ __forceinline__ int pair_tiles(int q_len, int ctx, int qp) {
  const int row0 = qp * kPrefillPairRows;
  const int nq = row0 + kPrefillPairRows / 2 < q_len ? 2 : 1;
  const int kv_end = min(ctx - q_len + row0 + nq * (kPrefillPairRows / 2), ctx);
  return (kv_end + 127) / 128;
}

struct RowInfo {
  int q_len, ctx;
  bool bad;
};

// The step's sizes: the host's, or (when AttnArgs::dims is set) the device's,
// checked against the host capacities.
struct StepSizes {
  int num_seqs, num_tokens, max_q_len, max_context_len;
};

__device__ __forceinline__ RowInfo row_info(const AttnArgs& a, const StepSizes& z, int s) {
  RowInfo r;
  const int c0 = a.cu_seqlens_q[s];
  const int c1 = a.cu_seqlens_q[s + 1];
  r.q_len = c1 - c0;
  r.ctx = a.context_lens[s];
  r.bad = r.q_len < 1 || r.ctx < r.q_len || r.ctx > z.max_context_len || r.q_len > z.max_q_len || c0 < 0 ||
          c1 > z.num_tokens || (int64_t(r.ctx) + a.block_size - 1) / a.block_size > a.max_blocks_per_seq;
  if (a.pad_lens && !r.bad) {
    const int pad = a.pad_lens[s];
    r.bad = pad < 0 || pad >= r.q_len;           // a chunk keeps at least one real row
  }
  return r;
}

// Stable-enough counting sort of n items into `out`, largest key first (keys
// at or above the last bucket share it).  Block-wide; contains __syncthreads.
template <typename Key>
__device__ void sort_desc(const int2* in, int2* out, int n, Key key, uint32_t* bucket, uint64_t* warp_sums) {
  if (n <= 1) {
    if (n == 1 && threadIdx.x == 0) out[0] = in[0];
    return;
  }
  for (int i = threadIdx.x; i < kCostBuckets; i += kPlanThreads) bucket[i] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += kPlanThreads) atomicAdd(&bucket[min(key(in[i]), kCostBuckets - 1)], 1u);
  __syncthreads();
  // descending order: thread t owns the kPer buckets just below kCostBuckets - kPer * t
  constexpr int kPer = kCostBuckets / kPlanThreads;
  uint32_t local[kPer], sum = 0;
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    local[k] = bucket[kCostBuckets - 1 - (threadIdx.x * kPer + k)];
    sum += local[k];
  }
  uint64_t total;
  uint32_t run = uint32_t(block_excl_scan(sum, warp_sums, total));
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    bucket[kCostBuckets - 1 - (threadIdx.x * kPer + k)] = run;
    run += local[k];
  }
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += kPlanThreads) {
    const int2 it = in[i];
    out[atomicAdd(&bucket[min(key(it), kCostBuckets - 1)], 1u)] = it;
  }
  __syncthreads();                          // `bucket` is reused by the next sort
}

__global__ void __launch_bounds__(kPlanThreads) plan_step_kernel(const AttnArgs a, const StepPlan p) {
  launch_dependents();                      // they wait for this grid on the device
  __shared__ uint64_t warp_sums[32];
  __shared__ uint32_t bucket[kCostBuckets];
  __shared__ int2 row_cache[kRowCache];     // (q_len, or 0 for a bad row; ctx)
  const int tid = threadIdx.x;
  StepSizes z = {a.num_seqs, a.num_tokens, a.max_q_len, a.max_context_len};
  if (a.dims) {
    z = StepSizes{a.dims[0], a.dims[1], a.dims[2], a.dims[3]};
    if (z.num_seqs < 0 || z.num_seqs > a.num_seqs || z.num_tokens < 0 || z.num_tokens > a.num_tokens ||
        z.max_q_len < 0 || z.max_q_len > a.max_q_len || z.max_context_len < 0 ||
        z.max_context_len > a.max_context_len) {
      if (tid == 0) raise_error(a.err, kErrInvalid);   // sizes beyond the capacities: an empty step
      z.num_seqs = 0;
    }
  }
  // (q_len, ctx) of row s after pass 1; q_len 0 marks a row left out
  auto row = [&](int s) -> int2 {
    if (s < kRowCache) return row_cache[s];
    const RowInfo r = row_info(a, z, s);
    return make_int2(r.bad ? 0 : r.q_len, r.ctx);
  };

  // Pass 1: check every row; total keys of the decode rows.
  uint64_t dec_keys = 0;
  int any_prefill = 0;
  for (int s = tid; s < z.num_seqs; s += kPlanThreads) {
    const RowInfo r = row_info(a, z, s);
    if (s < kRowCache) row_cache[s] = make_int2(r.bad ? 0 : r.q_len, r.ctx);
    if (r.bad)
      raise_error(a.err, kErrInvalid);
    else if (r.q_len == 1)
      dec_keys += uint64_t(r.ctx);
    else
      any_prefill = 1;
  }
  const bool decode_only = __syncthreads_or(any_prefill) == 0;
  uint64_t total_keys;
  block_excl_scan(dec_keys, warp_sums, total_keys);
  // Keys per decode split: every split pays a fixed cost (its merge, a
  // partial result written and read back, the pipeline fill of a new unit),
  // so splits are as long as possible while a split stays within 1/u of a
  // decode CTA's average share (total keys x groups of query heads / CTAs),
  // u = dec_units_per_cta: greedy claiming, longest unit first, then ends
  // every CTA within about one unit of the others.
  const uint64_t groups = uint64_t(p.dec_groups > 0 ? p.dec_groups : a.num_heads);
  const float per_cta = fmaxf(p.dec_units_per_cta[decode_only ? 0 : 1], 0.125f);
  const uint64_t target = uint64_t(ceilf(float(p.dec_ctas > 0 ? p.dec_ctas : 1) * per_cta));
  const uint64_t want = (total_keys * groups + target - 1) / target;
  const uint64_t per = want < uint64_t(kSplitKeys) ? uint64_t(kSplitKeys) : want;
  const uint64_t rounded = (per + kSplitKeys - 1) / kSplitKeys * kSplitKeys;
  const int split = rounded > (uint64_t(1) << 30) ? (1 << 30) : int(rounded);

  // Pass 2: list the items (unsorted).
  uint64_t base = 0;                        // items so far: decode in the low, prefill in the high word
  for (int s0 = 0; s0 < z.num_seqs; s0 += kPlanThreads) {
    const int s = s0 + tid;
    uint32_t nd = 0, np = 0, pairs = 0;     // decode items; prefill records (0 or 1) and their pairs
    if (s < z.num_seqs) {
      const int2 r = row(s);
      if (r.x > 0) {
        if (r.x == 1) {
          nd = uint32_t((r.y + split - 1) / split);
        } else {
          np = 1;
          pairs = uint32_t((r.x + kPrefillPairRows - 1) / kPrefillPairRows);
        }
      }
    }
    uint64_t total;
    const uint64_t off = base + block_excl_scan(uint64_t(nd) | (uint64_t(np) << 32), warp_sums, total);
    base += total;
    const uint32_t od = uint32_t(off), op = uint32_t(off >> 32);
    if (nd > 0) {
      if (od + nd <= uint32_t(p.dec_cap)) {
        for (uint32_t k = 0; k < nd; ++k) p.dec_scratch[od + k] = make_int2(s, int(k));
      } else {
        raise_error(a.err, kErrInvalid);
      }
    }
    if (np > 0) {
      if (op < uint32_t(p.pre_cap))
        p.pre_scratch[op] = make_int2(s, int(pairs));
      else
        raise_error(a.err, kErrInvalid);      // overlapping query ranges (malformed cu_seqlens_q)
    }
  }
  const int n_dec = min(int(uint32_t(base)), p.dec_cap);
  const int n_chunks = min(int(uint32_t(base >> 32)), p.pre_cap);
  // split tickets start at zero (coalesced over the whole [num_seqs][H] array)
  for (int i = tid; i < z.num_seqs * a.num_heads; i += kPlanThreads) p.tickets[i] = 0;
  __syncthreads();                          // every thread's items are written before any is re-read

  // Longest first, so that greedy claiming ends on short units.
  sort_desc(p.dec_scratch, p.dec_items, n_dec,
            [&](int2 it) {
              const int len = min(row(it.x).y - it.y * split, split);
              return (len + 15) / 16;
            },
            bucket, warp_sums);
  // Prefill: chunks by total cost, costliest first; then within a chunk all
  // units of one head together (its query pairs share that head's K/V tiles
  // in L2 while they run), costliest pair first.
  sort_desc(p.pre_scratch, p.pre_seqs, n_chunks,
            [&](int2 rec) {
              const int2 r = row(rec.x);
              int cost = 0;
              for (int qp = 0; qp < rec.y; ++qp) cost += pair_cost(r.x, r.y, qp);
              return cost;
            },
            bucket, warp_sums);
  const int unit_cap = p.pre_cap * a.num_heads;
  uint64_t unit_base = 0;                   // first unit of each sorted chunk, into pre_scratch[].x
  uint64_t pre_cost = 0;                    // sum of unit costs (KV tiles x query tiles) over all heads
  for (int c0 = 0; c0 < n_chunks; c0 += kPlanThreads) {
    const int c = c0 + tid;
    uint32_t n = 0, cost = 0;
    if (c < n_chunks) {
      const int2 rec = p.pre_seqs[c];
      const int2 r = row(rec.x);
      n = uint32_t(rec.y) * uint32_t(a.num_heads);
      for (int qp = 0; qp < rec.y; ++qp) cost += uint32_t(pair_cost(r.x, r.y, qp));
      const uint64_t all_heads = uint64_t(cost) * uint64_t(a.num_heads);
      cost = all_heads < 0x7FFFFFFFull ? uint32_t(all_heads) : 0x7FFFFFFFu;
    }
    uint64_t total;
    const uint64_t off = unit_base + block_excl_scan(uint64_t(n) | (uint64_t(cost) << 32), warp_sums, total);
    unit_base += uint64_t(uint32_t(total));
    pre_cost += total >> 32;
    const uint64_t off_units = uint32_t(off);
    if (c < n_chunks) p.pre_scratch[c] = make_int2(off_units < uint64_t(unit_cap) ? int(off_units) : unit_cap, 0);
  }
  if (unit_base > uint64_t(unit_cap) && tid == 0) raise_error(a.err, kErrInvalid);
  const int n_pre_units = int(unit_base < uint64_t(unit_cap) ? unit_base : uint64_t(unit_cap));
  // SMs for prefill in a mixed step: prefill on k SMs and decode on the rest
  // run side by side; each thread scores one k (k = tid + 1), the block keeps
  // the best (estimated step time, then the smaller k)
  int k = p.num_sms;
  {
    const float dec_bytes = float(total_keys) * float(p.kv_bytes_per_key);
    if (p.split_sms && n_pre_units > 0 && dec_bytes > 0.f && p.num_sms > 1) {
      const float pre_us = float(n_pre_units) * kPrefillUsPerUnit + float(pre_cost) * kPrefillUsPerCost;  // one SM
      const float serial = __fdividef(pre_us, float(p.num_sms)) +
                           __fdividef(dec_bytes, fminf(kDecodeBytesPerUs, p.dec_bytes_per_us_per_sm * p.num_sms));
      float score = 3.0e38f;
      const int kk = tid + 1;
      if (kk < p.num_sms) {
        const float bw = fminf(kDecodeBytesPerUs, p.dec_bytes_per_us_per_sm * float(p.num_sms - kk));
        score = fmaxf(__fdividef(pre_us, float(kk)), __fdividef(dec_bytes, bw));
      }
      // (score, k) minimum: scores are positive floats, so their bits order like the floats
      uint64_t key = (uint64_t(__float_as_uint(score)) << 32) | uint32_t(kk);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const uint64_t other = __shfl_xor_sync(0xffffffffu, key, o);
        key = other < key ? other : key;
      }
      if ((tid & 31) == 0) warp_sums[tid >> 5] = key;
      __syncthreads();
      uint64_t best = warp_sums[0];
      for (int w = 1; w < kPlanThreads / 32; ++w) best = warp_sums[w] < best ? warp_sums[w] : best;
      if (__uint_as_float(uint32_t(best >> 32)) < kSplitGain * serial) k = int(uint32_t(best));
    }
  }

  // Segments: the length L (KV tiles), then each chunk's entries with it
  // (pre_scratch[c].y: first entry of chunk c); segments are kept only if
  // some pair is cut and their partial slots fit
  int seg = 0;
  if (p.pre_partials && n_pre_units > 0) {
    const float pre_us = float(n_pre_units) * kPrefillUsPerUnit + float(pre_cost) * kPrefillUsPerCost;
    const float dec_us = __fdividef(float(total_keys) * float(p.kv_bytes_per_key), p.dec_bytes_per_us_per_sm);
    // an SM's share in KV tiles of a two-tile unit
    const float share = __fdividef(pre_us + dec_us, float(p.num_sms) * 2.0f * kPrefillUsPerCost);
    const float want = ceilf(__fdividef(share, float(kSegPerShare)));
    seg = want < float(kSegMinTiles) ? kSegMinTiles : (want > 65535.0f ? 65535 : int(want));
  }
  uint64_t n_entries = n_pre_units;
  if (seg > 0) {
    uint64_t entry_base = 0;
    for (int c0 = 0; c0 < n_chunks; c0 += kPlanThreads) {
      const int c = c0 + tid;
      uint32_t e = 0;
      if (c < n_chunks) {
        const int2 rec = p.pre_seqs[c];
        const int2 r = row(rec.x);
        for (int qp = 0; qp < rec.y; ++qp) e += uint32_t((pair_tiles(r.x, r.y, qp) + seg - 1) / seg);
        e *= uint32_t(a.num_heads);
      }
      uint64_t total;
      const uint64_t off = entry_base + block_excl_scan(e, warp_sums, total);
      entry_base += total;
      if (c < n_chunks) p.pre_scratch[c].y = int(off < uint64_t(kPrefillSegSlots) ? off : kPrefillSegSlots);
    }
    if (entry_base > uint64_t(n_pre_units) && entry_base <= uint64_t(kPrefillSegSlots)) n_entries = entry_base;
    else seg = 0;                                          // no pair cut, or too many segments: whole units
  }
  for (int i = tid; i < int(seg > 0 ? n_entries * kSegTicketsPerSlot : 0); i += kPlanThreads) p.pre_tickets[i] = 0;
  __syncthreads();
  // One thread per unit (chunk, head, pair) writes the unit's entries: unit
  // u belongs to the last chunk starting at or before it.  Within a chunk
  // (and within a segment index) the order is one of two:
  //  * head by head, costliest pair first, when decode rows share the step:
  //    the pairs of one head then stream the same K/V together, read once
  //    from HBM, which the decode beside them saturates;
  //  * costliest pair first over all heads, then the next pair, in a
  //    prefill-only step where the units differ in size: greedy claiming
  //    then takes the longest units first and ends on short ones (measured
  //    on GB300: a 2048-token chunk at p = 0 in 0.069 against 0.086 ms, the
  //    32768-token prompt in 16 chunks 7.68 against 7.91 ms; the mixed step
  //    with 64 decode rows 0.439 against 0.420 ms in this order, hence the
  //    first one there).
  const bool pair_major = n_dec == 0;
  for (int u = tid; u < n_pre_units; u += kPlanThreads) {
    int lo = 0, hi = n_chunks - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.pre_scratch[mid].x <= u) lo = mid; else hi = mid - 1;
    }
    const int2 rec = p.pre_seqs[lo];
    const int2 r = row(rec.x);
    const int np = rec.y;
    const int local = u - p.pre_scratch[lo].x;
    // pair-major only where unit sizes differ enough to matter (a causal
    // chunk's first pairs are short): a head's pairs read the same keys, and
    // head by head they do so together, once from HBM
    const bool pm = pair_major && 2 * pair_tiles(r.x, r.y, 0) < pair_tiles(r.x, r.y, np - 1);
    const int h = pm ? local % a.num_heads : local / np;
    const int qp = pm ? np - 1 - local / a.num_heads : np - 1 - (local - h * np);
    const int nt = pair_tiles(r.x, r.y, qp);
    if (seg == 0) {
      p.pre_units[u] = make_int4(rec.x, qp | (h << 16), nt << 16, -1);
      continue;
    }
    // Segments: by segment index kk (all heads, then the next index), then
    // in the order above.  Pairs later in the chunk have more tiles, so the
    // cnt pairs with a segment kk are the last ones.  A pair's segments share
    // its slots [slot0, slot0 + nseg).
    int per_head = 0, before = 0;
    for (int q2 = 0; q2 < np; ++q2) {
      const int ns = (pair_tiles(r.x, r.y, q2) + seg - 1) / seg;
      per_head += ns;
      if (q2 < qp) before += ns;
    }
    const int e_c = p.pre_scratch[lo].y;
    const int nseg = (nt + seg - 1) / seg;
    const int slot0 = nseg > 1 ? e_c + h * per_head + before : -1;
    int off = 0;
    for (int kk = 0; kk < nseg; ++kk) {
      int cnt = 0;
      for (int q2 = 0; q2 < np; ++q2) cnt += pair_tiles(r.x, r.y, q2) > kk * seg ? 1 : 0;
      const int j0 = kk * seg, j1 = min(j0 + seg, nt);
      // a group of whole segments keeps the head-by-head order; a group of
      // last segments (sizes differ: its first pair is the shortest) may go
      // pair-major
      const bool pm_kk = pair_major && pair_tiles(r.x, r.y, np - cnt) < j0 + seg;
      const int pos = pm_kk ? (np - 1 - qp) * a.num_heads + h : h * cnt + (np - 1 - qp);
      p.pre_units[e_c + off + pos] = make_int4(rec.x, qp | (h << 16), j0 | (j1 << 16), slot0);
      off += cnt * a.num_heads;
    }
  }
  if (tid == 0) {
    p.header[0] = n_dec;
    p.header[1] = int(n_entries);
    p.header[2] = 0;
    p.header[3] = 0;
    p.header[4] = int32_t(p.tag);
    p.header[5] = split;
    p.header[6] = z.num_seqs;
    p.header[7] = z.num_tokens;
    p.header[8] = k;
    p.header[9] = seg;
    p.header[10] = 0;                     // prefill CTAs done claiming
    p.header[11] = 0;                     // decode CTAs done claiming
  }
}

}  // namespace

size_t step_workspace_bytes(int32_t num_seqs, int32_t num_tokens, int32_t num_heads, int32_t head_dim,
                            int32_t max_context_len) {
  const size_t S = size_t(num_seqs > 0 ? num_seqs : 0), T = size_t(num_tokens > 0 ? num_tokens : 0);
  const size_t splits = size_t((max_context_len + kSplitKeys - 1) / kSplitKeys);
  const size_t pre_cap = T / kPrefillPairRows + (S < T / 2 ? S : T / 2) + 1;
  return 256 +                                                        // header
         2 * align256(S * splits * sizeof(int2)) +                    // decode items + scratch
         2 * align256(pre_cap * sizeof(int2)) +                       // prefill chunk records + scratch
         align256((pre_cap * num_heads + kPrefillSegSlots) * sizeof(int4)) +   // prefill entries
         align256(size_t(kPrefillSegSlots) * kSegTicketsPerSlot * sizeof(int32_t)) +   // segment tickets
         (has_seg_partials(S, T, max_context_len)                     // prefill segment partials
              ? size_t(kPrefillSegSlots) * kPrefillPairRows * (head_dim + 2) * sizeof(float)
              : 0) +
         align256(S * num_heads * sizeof(int32_t)) +                  // tickets
         (splits > 1 ? S * num_heads * splits * (head_dim + 2) * sizeof(float) : 0);   // partials
}

cb_status step_plan_layout(void* workspace, size_t workspace_bytes, int32_t num_seqs, int32_t num_tokens,
                           int32_t num_heads, int32_t head_dim, int32_t max_context_len, StepPlan* plan) {
  const size_t need = step_workspace_bytes(num_seqs, num_tokens, num_heads, head_dim, max_context_len);
  if (!workspace || workspace_bytes < need)
    return fail(CB_ERR_INVALID, "workspace too small: %zu bytes given, %zu needed", workspace_bytes, need);
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
    return fail(CB_ERR_INVALID, "workspace must be 256-byte aligned");
  const size_t S = size_t(num_seqs), T = size_t(num_tokens);
  const size_t splits = size_t((max_context_len + kSplitKeys - 1) / kSplitKeys);
  const size_t pre_cap = T / kPrefillPairRows + (S < T / 2 ? S : T / 2) + 1;
  char* w = static_cast<char*>(workspace);
  plan->header = reinterpret_cast<int32_t*>(w);
  w += 256;
  plan->dec_items = reinterpret_cast<int2*>(w);
  w += align256(S * splits * sizeof(int2));
  plan->dec_scratch = reinterpret_cast<int2*>(w);
  w += align256(S * splits * sizeof(int2));
  plan->pre_seqs = reinterpret_cast<int2*>(w);
  w += align256(pre_cap * sizeof(int2));
  plan->pre_scratch = reinterpret_cast<int2*>(w);
  w += align256(pre_cap * sizeof(int2));
  plan->pre_units = reinterpret_cast<int4*>(w);
  w += align256((pre_cap * num_heads + kPrefillSegSlots) * sizeof(int4));
  plan->pre_tickets = reinterpret_cast<int32_t*>(w);
  w += align256(size_t(kPrefillSegSlots) * kSegTicketsPerSlot * sizeof(int32_t));
  plan->pre_partials = nullptr;
  if (has_seg_partials(S, T, max_context_len)) {
    plan->pre_partials = reinterpret_cast<float*>(w);
    w += size_t(kPrefillSegSlots) * kPrefillPairRows * (head_dim + 2) * sizeof(float);
  }
  plan->tickets = reinterpret_cast<int32_t*>(w);
  w += align256(S * num_heads * sizeof(int32_t));
  plan->partials = reinterpret_cast<float*>(w);
  plan->max_splits = int32_t(splits);
  plan->dec_cap = int32_t(S * splits);
  plan->pre_cap = int32_t(pre_cap);
  plan->dec_ctas = 0;
  plan->dec_groups = 0;
  plan->num_sms = sm_count();
  plan->kv_bytes_per_key = 0;
  plan->dec_bytes_per_us_per_sm = 9.0e4f;
  plan->split_sms = 0;
  static std::atomic<uint32_t> next_tag{1};
  plan->tag = next_tag.fetch_add(1);
  return CB_OK;
}

cb_status launch_plan(const AttnArgs& a, const StepPlan& plan, cudaStream_t stream) {
  NvtxRange nvtx("cb.plan");
  plan_step_kernel<<<1, kPlanThreads, 0, stream>>>(a, plan);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "step plan: launch");
  return CB_OK;
}

}  // namespace cb
