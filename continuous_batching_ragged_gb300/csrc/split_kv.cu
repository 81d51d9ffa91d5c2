// K2 + K4: split-KV attention of single query rows on CUDA cores, merged by
// log-sum-exp.
//
// Page "continuous-batching" (zhangchitc.github.io), sections "Ragged
// batching" (a decoding request's one query is dotted with every key it has
// seen, cache plus its new token) and "Inside the kernel" (the request's cache
// is read one paged block at a time; each block's scores weight its values and
// are accumulated into a running state -- online softmax).
//
// Decode is HBM-bound (one multiply-add per key byte pair), so the design
// goal is bytes in flight, not arithmetic:
//   * grid (split, head, row): a row's keys are cut into fixed 512-key splits,
//     so a long context spreads over many CTAs;
//   * 4 warps per CTA, each warp walks 16-key tiles; a lane handles one
//     16-byte chunk of a key row, half a warp covers one 256-byte row;
//   * bf16, head_dim 128, block size a multiple of 16 (the decode workload):
//     a 16-key tile of one head is one contiguous 4 KB chunk of the paged pool
//     for K and one for V, so each warp streams its tiles with 1-D bulk async
//     copies (cp.async.bulk) into a private 3-stage shared-memory ring, three
//     tiles ahead of its arithmetic; other shapes load straight to registers;
//   * the 16-lane dot-product reduction is a transpose-reduce (each shuffle
//     step halves the rows a lane holds), 8 shuffles for 8 rows instead of 32;
//   * running max / sum / accumulator per warp, merged across warps in shared
//     memory, then across splits by the last CTA of the row to finish (an
//     atomic ticket), which writes the output row.
#include <algorithm>
#include <mutex>
#include <cfloat>

#include "device_common.cuh"
#include "kernels.h"
#include "runtime.h"
#include "sm100_ptx.cuh"

namespace cb {
namespace {

constexpr int kWarps = 4;
constexpr int kTile = 16;     // keys per warp iteration
constexpr int kStages = 3;    // bulk-copy ring depth per warp
constexpr uint32_t kTileBytes = kTile * 128 * 2;   // one bf16 16 x 128 K (or V) tile: 4 KB
// Decode units per persistent CTA that the step plan's split length aims
// for, in a decode-only step [0] and beside prefill chunks [1], for this
// kernel and for the tensor-core one, whose units pay more at each start
// (the query rows, the first tiles and the merge of every split).
constexpr float kUnitsPerCta[2] = {2.f, 6.f};
constexpr float kTcUnitsPerCta[2] = {1.f, 1.f};
constexpr float kTcUnitsPerCtaWide = 0.75f;   // groups of more than 16 heads (MQA at 32 heads)

struct SplitArgs {
  AttnArgs a;
  float* partials;          // [rows][H][max_splits][A + 2]
  int32_t* tickets;         // [rows][H]
  int32_t max_splits;
  const int2* items;        // persistent decode: the plan's (sequence, split) items
  const int32_t* header;    // persistent decode: [0] = number of items
  int32_t* claims;          // persistent decode: claim counter
  int32_t* done;            // persistent decode: CTAs done claiming (the last resets both)
  int32_t item_cap;         // persistent decode: capacity of the item list
  uint32_t tag;             // persistent decode: the plan's call tag
  int32_t n_groups;         // persistent decode: units per item (query-head groups)
  int32_t wait_previous;    // persistent decode: wait for the kernel launched before (the plan)
};

// Packed fp32 pairs (Blackwell f32x2 FMA): two FMAs per instruction.
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpk2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sum v[0..N) over the LPR lanes of a row group so that, afterwards, v[0] of
// lane l holds the full sum of row index  sum_k ((l & (LPR >> k)) ? (N >> k) : 0).
template <int N, int LPR>
__device__ __forceinline__ void transpose_reduce(float (&v)[N], int lane) {
  int cnt = N;
#pragma unroll
  for (int bit = LPR / 2; bit >= 1; bit >>= 1) {
    if (cnt > 1) {
      const int half = cnt / 2;
      const bool upper = lane & bit;
#pragma unroll
      for (int i = 0; i < N / 2; ++i) {
        if (i < half) {
          const float send = upper ? v[i] : v[i + half];
          const float keep = upper ? v[i + half] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, bit);
        }
      }
      cnt = half;
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], bit);
    }
  }
}

// Which query row this CTA serves and which of its keys [k0, k1).
struct RowPlan {
  int s, t, nsplit, k0, k1;
};

template <bool ROW_MODE>
__device__ __forceinline__ bool plan_row(const AttnArgs& a, int split, int h, RowPlan& pl) {
  int s, t;
  if (ROW_MODE) {
    t = blockIdx.z;
    int lo = 0, hi = a.num_seqs - 1;
    while (lo < hi) {                     // last s with cu[s] <= t
      const int mid = (lo + hi + 1) >> 1;
      if (a.cu_seqlens_q[mid] <= t) lo = mid; else hi = mid - 1;
    }
    s = lo;
  } else {
    s = blockIdx.z;
  }
  const int c0 = a.cu_seqlens_q[s];
  const int c1 = a.cu_seqlens_q[s + 1];
  const int q_len = c1 - c0;
  const int ctx = a.context_lens[s];
  if (!ROW_MODE) {
    if (q_len > 1) return false;          // prefill chunk: not ours
    t = c0;
  }
  const bool bad = q_len < 1 || ctx < q_len || ctx > a.max_context_len || q_len > a.max_q_len ||
                   c0 < 0 || c1 > a.num_tokens || (ROW_MODE && (t < c0 || t >= c1)) ||
                   (ctx + a.block_size - 1) / a.block_size > a.max_blocks_per_seq;
  if (bad) {
    if (split == 0 && h == 0 && threadIdx.x == 0) raise_error(a.err, kErrInvalid);
    return false;
  }
  const int key_end = ROW_MODE ? ctx - q_len + (t - c0) + 1 : ctx;
  pl.s = s;
  pl.t = t;
  pl.nsplit = (key_end + kSplitKeys - 1) / kSplitKeys;
  if (split >= pl.nsplit) return false;
  pl.k0 = split * kSplitKeys;
  pl.k1 = min(key_end, pl.k0 + kSplitKeys);
  return true;
}

// Shared scratch of the split epilogue.
template <int A>
struct MergeSmem {
  float acc[kWarps][A];
  float m[kWarps], l[kWarps];
  int last;
};

// Combine the warps' (m, l, acc) of this split, then either write the output
// row (one split) or publish the partial and, in the last CTA of the row to
// finish, merge all partials by log-sum-exp.
template <typename T, int A, bool ROW_MODE, int EPV, int LPR>
__device__ __forceinline__ void finish_split(const SplitArgs& sa, const RowPlan& pl, int split, int h,
                                             float m_run, float l_run, float (&acc)[EPV],
                                             MergeSmem<A>& sm) {
  const AttnArgs& a = sa.a;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int g = lane / LPR, c = lane % LPR;
  // lanes of different row groups hold the same chunk: add them
#pragma unroll
  for (int o = LPR; o < 32; o <<= 1) {
#pragma unroll
    for (int e = 0; e < EPV; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], o);
  }
  if (g == 0) {
#pragma unroll
    for (int e = 0; e < EPV; ++e) sm.acc[warp][c * EPV + e] = acc[e];
  }
  if (lane == 0) {
    sm.m[warp] = m_run;
    sm.l[warp] = l_run;
  }
  __syncthreads();

  const int d = threadIdx.x;
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm.m[w]);
  float L = 0.f, o = 0.f;
  if (d < A) {
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float f = ex2(sm.m[w] - M);   // a warp with no keys has m = -inf: weight 0
      L = fmaf(sm.l[w], f, L);
      o = fmaf(sm.acc[w][d], f, o);
    }
  }
  T* out_row = static_cast<T*>(a.out) + (size_t(pl.t) * a.num_heads + h) * A;
  if (pl.nsplit == 1) {
    if (d < A) store1(out_row + d, o / L);
    return;
  }
  const int row_id = ROW_MODE ? pl.t : pl.s;
  float* part = sa.partials + ((size_t(row_id) * a.num_heads + h) * sa.max_splits) * (A + 2);
  if (d < A) part[size_t(split) * (A + 2) + d] = o;
  if (d == 0) {
    part[size_t(split) * (A + 2) + A] = M;
    part[size_t(split) * (A + 2) + A + 1] = L;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    int32_t* ticket = sa.tickets + size_t(row_id) * a.num_heads + h;
    sm.last = atomicAdd(ticket, 1) == pl.nsplit - 1;
    if (sm.last) *ticket = 0;             // every split has arrived: reset for the next call
  }
  __syncthreads();
  if (!sm.last) return;
  __threadfence();
  if (d < A) {
    float MM = -INFINITY;
    for (int k = 0; k < pl.nsplit; ++k) MM = fmaxf(MM, __ldcg(part + size_t(k) * (A + 2) + A));
    float LL = 0.f, oo = 0.f;
    for (int k = 0; k < pl.nsplit; ++k) {
      const float* pk = part + size_t(k) * (A + 2);
      const float f = ex2(__ldcg(pk + A) - MM);
      LL = fmaf(__ldcg(pk + A + 1), f, LL);
      oo = fmaf(__ldcg(pk + d), f, oo);
    }
    store1(out_row + d, oo / LL);
  }
}

// One 16-key tile of the online softmax: scores of the lane's NR rows from
// kv[], running max/sum update, accumulate p * v into acc.
template <typename T, int EPV, int LPR, int RPL, int NR>
__device__ __forceinline__ void tile_update(const float (&qf)[EPV], const uint4 (&kv)[NR], const uint4 (&vv)[NR],
                                            int base, int k1, int lane, float& m_run, float& l_run,
                                            float (&acc)[EPV]) {
  const int g = lane / LPR, c = lane % LPR;
  float sc[NR];
#pragma unroll
  for (int i = 0; i < NR; ++i) {
    float kf[EPV];
    Vec16<T>::to_float(kv[i], kf);
    float d = 0.f;
#pragma unroll
    for (int e = 0; e < EPV; ++e) d = fmaf(qf[e], kf[e], d);
    sc[i] = d;
  }
  transpose_reduce<NR, LPR>(sc, lane);
  // lane holds the score of tile row g + RPL * idx, idx = (lane % LPR) / (LPR / NR)
  const int idx = c / (LPR / NR);
  const int my_row = base + g + RPL * idx;
  const float sv = my_row < k1 ? sc[0] : -INFINITY;
  const float m_new = fmaxf(m_run, warp_max(sv));
  const float alpha = ex2(m_run - m_new);
  const float pr = ex2(sv - m_new);
  const float psum = warp_sum((c % (LPR / NR)) == 0 ? pr : 0.f);
  l_run = l_run * alpha + psum;
#pragma unroll
  for (int e = 0; e < EPV; ++e) acc[e] *= alpha;
#pragma unroll
  for (int i = 0; i < NR; ++i) {
    const float pi = __shfl_sync(0xffffffffu, pr, g * LPR + i * (LPR / NR));
    float vf[EPV];
    Vec16<T>::to_float(vv[i], vf);
#pragma unroll
    for (int e = 0; e < EPV; ++e) acc[e] = fmaf(pi, vf[e], acc[e]);
  }
  m_run = m_new;
}

// tile_update for the GU query heads of one key/value head: each K and V row
// is converted to fp32 once for all GU heads, the dot products and P V
// updates run two lanes of work per packed f32x2 FMA, and two per-tile
// reductions go:
//  * the running max m_run (warp-uniform) moves only when some score of the
//    tile exceeds it by more than 8 in the exp2 domain (one vote; the warp
//    max and the rescale run only then), so p stays below 2^8;
//  * l_run is this lane's partial row sum (each row counted by one lane of
//    its pair), summed over the warp once per unit, before the merge.
template <int GU, int EPV, int LPR, int RPL, int NR>
__device__ __forceinline__ void group_tile_update(const float (&qf)[GU][EPV], const uint4 (&kv)[NR],
                                                  const uint4 (&vv)[NR], int base, int k1, int lane,
                                                  float (&m_run)[GU], float (&l_run)[GU], float (&acc)[GU][EPV]) {
  using T = __nv_bfloat16;
  const int g = lane / LPR, c = lane % LPR;
  float sc[GU][NR];
#pragma unroll
  for (int i = 0; i < NR; ++i) {
    float kf[EPV];
    Vec16<T>::to_float(kv[i], kf);
#pragma unroll
    for (int hh = 0; hh < GU; ++hh) {
      uint64_t d2 = pk2(0.f, 0.f);
#pragma unroll
      for (int e = 0; e < EPV; e += 2) d2 = fma2(pk2(qf[hh][e], qf[hh][e + 1]), pk2(kf[e], kf[e + 1]), d2);
      float d0, d1;
      unpk2(d2, d0, d1);
      sc[hh][i] = d0 + d1;
    }
  }
  const int idx = c / (LPR / NR);
  const int my_row = base + g + RPL * idx;
  float pr[GU];
#pragma unroll
  for (int hh = 0; hh < GU; ++hh) {
    transpose_reduce<NR, LPR>(sc[hh], lane);
    const float sv = my_row < k1 ? sc[hh][0] : -INFINITY;
    if (__any_sync(0xffffffffu, sv > m_run[hh] + 8.0f)) {
      const float m_new = fmaxf(m_run[hh], warp_max(sv));
      const float alpha = ex2(m_run[hh] - m_new);
      l_run[hh] *= alpha;
#pragma unroll
      for (int e = 0; e < EPV; ++e) acc[hh][e] *= alpha;
      m_run[hh] = m_new;
    }
    pr[hh] = ex2(sv - m_run[hh]);
    if ((c % (LPR / NR)) == 0) l_run[hh] += pr[hh];
  }
#pragma unroll
  for (int i = 0; i < NR; ++i) {
    float vf[EPV];
    Vec16<T>::to_float(vv[i], vf);
#pragma unroll
    for (int hh = 0; hh < GU; ++hh) {
      const float pi = __shfl_sync(0xffffffffu, pr[hh], g * LPR + i * (LPR / NR));
      const uint64_t pi2 = pk2(pi, pi);
#pragma unroll
      for (int e = 0; e < EPV; e += 2) {
        const uint64_t a2 = fma2(pi2, pk2(vf[e], vf[e + 1]), pk2(acc[hh][e], acc[hh][e + 1]));
        unpk2(a2, acc[hh][e], acc[hh][e + 1]);
      }
    }
  }
}

template <typename T, int A>
__device__ __forceinline__ void load_q(const AttnArgs& a, int t, int h, int c, float (&qf)[Vec16<T>::N]) {
  constexpr int EPV = Vec16<T>::N;
  const uint4 qv = *reinterpret_cast<const uint4*>(static_cast<const T*>(a.q) + (size_t(t) * a.num_heads + h) * A +
                                                   c * EPV);
  Vec16<T>::to_float(qv, qf);
#pragma unroll
  for (int e = 0; e < EPV; ++e) qf[e] *= a.scale_log2;    // scores in the exp2 domain
}

// Loads straight to registers: any dtype, head_dim 64/128, any block size.
template <typename T, int A, bool ROW_MODE>
__global__ void __launch_bounds__(kWarps * 32) split_kv_kernel(const SplitArgs sa) {
  constexpr int EPV = Vec16<T>::N;        // elements per 16-byte load
  constexpr int LPR = A / EPV;            // lanes per key row
  constexpr int RPL = 32 / LPR;           // key rows per warp load
  constexpr int NR = kTile / RPL;         // key rows per lane per tile
  static_assert(NR <= LPR && NR >= 1, "tile shape");
  const AttnArgs& a = sa.a;
  const int split = blockIdx.x, h = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  RowPlan pl;
  if (!plan_row<ROW_MODE>(a, split, h, pl)) return;
  const int g = lane / LPR, c = lane % LPR;
  float qf[EPV];
  load_q<T, A>(a, pl.t, h, c, qf);

  const T* kp = static_cast<const T*>(a.k_pool);
  const T* vp = static_cast<const T*>(a.v_pool);
  const int32_t* bt = a.block_tables + size_t(pl.s) * a.max_blocks_per_seq;
  const int B = a.block_size;
  const size_t head_off = size_t(h) * B * A;
  const size_t blk_stride = size_t(a.num_heads) * B * A;
  const bool whole_tiles = (B % kTile) == 0;
  float m_run = -INFINITY, l_run = 0.f;
  float acc[EPV];
#pragma unroll
  for (int e = 0; e < EPV; ++e) acc[e] = 0.f;

  for (int base = pl.k0 + warp * kTile; base < pl.k1; base += kWarps * kTile) {
    uint4 kv[NR], vv[NR];
    int32_t tile_blk = 0;
    if (whole_tiles) {
      tile_blk = bt[base / B];
      if (tile_blk < 0 || tile_blk >= a.num_blocks) {
        if (lane == 0) raise_error(a.err, kErrBounds);
        tile_blk = -1;
      }
    }
#pragma unroll
    for (int i = 0; i < NR; ++i) {
      const int j = base + g + RPL * i;
      kv[i] = make_uint4(0, 0, 0, 0);
      vv[i] = make_uint4(0, 0, 0, 0);
      if (j < pl.k1) {
        int32_t blk = tile_blk;
        if (!whole_tiles) {
          blk = bt[j / B];
          if (blk < 0 || blk >= a.num_blocks) {
            raise_error(a.err, kErrBounds);
            blk = -1;
          }
        }
        if (blk >= 0) {
          const size_t off = size_t(blk) * blk_stride + head_off + size_t(j % B) * A + c * EPV;
          kv[i] = ldg_stream(kp + off);
          vv[i] = ldg_stream(vp + off);
        }
      }
    }
    tile_update<T, EPV, LPR, RPL, NR>(qf, kv, vv, base, pl.k1, lane, m_run, l_run, acc);
  }
  __shared__ MergeSmem<A> sm;
  finish_split<T, A, ROW_MODE, EPV, LPR>(sa, pl, split, h, m_run, l_run, acc, sm);
}

// One decode unit: (sequence, split, group of GU query heads sharing one KV
// head) and the keys [k0, k1) it covers.
struct Unit {
  int u;                      // claimed unit index; >= the unit count: no more work
  int s, t, grp, h0, hkv, split, nsplit, k0, k1;
};

// Shared scratch of the epilogue of a unit of GU query heads.
template <int GU>
struct GroupSmem {
  float acc[GU][kWarps][128];
  float m[GU][kWarps], l[GU][kWarps];
  int last;
};

// Combine the warps' (m, l, acc) of each of the unit's GU heads, then either
// write the output rows (one split) or publish the partials and, in the last
// CTA of the (sequence, group) to finish, merge every split by log-sum-exp.
template <int GU>
__device__ __forceinline__ void finish_group(const SplitArgs& sa, const Unit& U, const float (&m_run)[GU],
                                             const float (&l_run)[GU], float (&acc)[GU][8], GroupSmem<GU>& sm) {
  using T = __nv_bfloat16;
  constexpr int A = 128, EPV = 8, LPR = 16;
  const AttnArgs& a = sa.a;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int g = lane / LPR, c = lane % LPR;
#pragma unroll
  for (int hh = 0; hh < GU; ++hh) {
    // lanes of the two row groups hold the same chunk: add them
#pragma unroll
    for (int e = 0; e < EPV; ++e) acc[hh][e] += __shfl_xor_sync(0xffffffffu, acc[hh][e], LPR);
    if (g == 0) {
#pragma unroll
      for (int e = 0; e < EPV; ++e) sm.acc[hh][warp][c * EPV + e] = acc[hh][e];
    }
    if (lane == 0) {
      sm.m[hh][warp] = m_run[hh];
      sm.l[hh][warp] = l_run[hh];
    }
  }
  __syncthreads();
  const int d = threadIdx.x;                // one output dimension per thread (128 threads)
  const int H = a.num_heads;
  float* part0 = sa.partials + (size_t(U.s) * H * sa.max_splits) * (A + 2);
#pragma unroll
  for (int hh = 0; hh < GU; ++hh) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm.m[hh][w]);
    float L = 0.f, o = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float f = ex2(sm.m[hh][w] - M);   // a warp with no keys has m = -inf: weight 0
      L = fmaf(sm.l[hh][w], f, L);
      o = fmaf(sm.acc[hh][w][d], f, o);
    }
    const int h = U.h0 + hh;
    if (U.nsplit == 1) {
      store1(static_cast<T*>(a.out) + (size_t(U.t) * H + h) * A + d, o / L);
    } else {
      float* part = part0 + (size_t(h) * sa.max_splits + U.split) * (A + 2);
      part[d] = o;
      if (d == 0) {
        part[A] = M;
        part[A + 1] = L;
      }
    }
  }
  if (U.nsplit == 1) return;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    int32_t* ticket = sa.tickets + size_t(U.s) * sa.n_groups + U.grp;
    sm.last = atomicAdd(ticket, 1) == U.nsplit - 1;
    if (sm.last) *ticket = 0;             // every split has arrived: reset for the next call
  }
  __syncthreads();
  if (!sm.last) return;
  __threadfence();
#pragma unroll
  for (int hh = 0; hh < GU; ++hh) {
    const int h = U.h0 + hh;
    const float* part = part0 + size_t(h) * sa.max_splits * (A + 2);
    float MM = -INFINITY;
    for (int k = 0; k < U.nsplit; ++k) MM = fmaxf(MM, __ldcg(part + size_t(k) * (A + 2) + A));
    float LL = 0.f, oo = 0.f;
    for (int k = 0; k < U.nsplit; ++k) {
      const float* pk = part + size_t(k) * (A + 2);
      const float f = ex2(__ldcg(pk + A) - MM);
      LL = fmaf(__ldcg(pk + A + 1), f, LL);
      oo = fmaf(__ldcg(pk + d), f, oo);
    }
    store1(static_cast<T*>(a.out) + (size_t(U.t) * H + h) * A + d, oo / LL);
  }
}

__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <int GU>
constexpr uint32_t bulk_smem_bytes() {
  return kWarps * kStages * 2 * kTileBytes + kWarps * kStages * (8 + 4) + sizeof(GroupSmem<GU>) + 2 * sizeof(Unit);
}

// Decode rows, bf16, head_dim 128, block size a multiple of 16, persistent:
// a fixed grid of CTAs claims units (sequence, split, group of GU query heads
// that share one KV head -- GU = 1 for multi-head attention) from the step
// plan until none are left.  Each warp streams its 16-key K/V tiles (4 KB
// each, contiguous in the pool) with bulk async copies into a private
// kStages-deep shared ring, and every tile serves all GU heads of the unit.
// The ring runs across units: once a warp has issued the last tile of its
// current unit it goes on with the first tiles of the unit the CTA claimed
// next, so the copies of the next unit are in flight while the current one
// is merged and written.
template <int GU>
__global__ void __launch_bounds__(kWarps * 32, 2) split_kv_persistent_kernel(const SplitArgs sa) {
  using T = __nv_bfloat16;
  constexpr int A = 128, EPV = 8, LPR = 16, RPL = 2, NR = 8;
  const AttnArgs& a = sa.a;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane / LPR, c = lane % LPR;

  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem + warp * kStages * 2 * kTileBytes;                  // [stage][K | V]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kWarps * kStages * 2 * kTileBytes) + warp * kStages;
  int* valid = reinterpret_cast<int*>(smem + kWarps * kStages * 2 * kTileBytes + kWarps * kStages * 8) +
               warp * kStages;
  GroupSmem<GU>& sm = *reinterpret_cast<GroupSmem<GU>*>(smem + kWarps * kStages * 2 * kTileBytes +
                                                        kWarps * kStages * 8 + kWarps * kStages * 4);
  Unit* slots = reinterpret_cast<Unit*>(reinterpret_cast<uint8_t*>(&sm) + sizeof(GroupSmem<GU>));   // [2]
  __shared__ int abort_flag;
  if (lane == 0) {
    for (int st = 0; st < kStages; ++st) sm100::mbar_init(sm100::smem_u32(&bars[st]), 1);
    sm100::fence_mbar_init();
  }
  if (threadIdx.x == 0) abort_flag = 0;
  if (sa.wait_previous) grid_dependency_wait();   // the plan kernel has finished
  const int H = a.num_heads;                // query heads
  const int G = H / a.num_kv_heads;         // query heads per KV head
  const int n_groups = sa.n_groups;         // = H / GU
  const uint32_t seen_tag = uint32_t(__ldcg(sa.header + 4));
  const int n_items = __ldcg(sa.header);
  if (seen_tag != sa.tag || n_items < 0 || n_items > sa.item_cap || __ldcg(sa.header + 5) < kSplitKeys) {
    if (threadIdx.x == 0) raise_error(a.err, kErrInvalid);
    return;
  }
  const int n_units = n_items * n_groups;
  if (int(blockIdx.x) >= n_units) return;   // no unit could be left for this CTA
  const int split_keys = __ldcg(sa.header + 5);            // keys per split, chosen by the plan
  const T* kp = static_cast<const T*>(a.k_pool);
  const T* vp = static_cast<const T*>(a.v_pool);
  const int B = a.block_size;
  const size_t blk_stride = size_t(a.num_kv_heads) * B * A;

  // one thread: claim the next unit and describe it in `slot`
  auto claim = [&](Unit& slot) {
    Unit U;
    U.u = abort_flag ? n_units : atomicAdd(sa.claims, 1);
    if (U.u < n_units) {
      const int2 it = __ldcg(sa.items + U.u / n_groups);
      U.grp = U.u % n_groups;
      U.h0 = U.grp * GU;
      U.hkv = U.h0 / G;
      U.s = it.x;
      U.split = it.y;
      bool bad = U.s < 0 || U.s >= a.num_seqs || U.split < 0;
      int ctx = 0;
      if (!bad) {
        U.t = __ldcg(a.cu_seqlens_q + U.s);
        ctx = __ldcg(a.context_lens + U.s);
        U.nsplit = (ctx + split_keys - 1) / split_keys;
        bad = U.t < 0 || U.t >= a.num_tokens || ctx < 1 || ctx > a.max_context_len || U.split >= U.nsplit;
      }
      if (bad) {                            // never happens with a plan from this call
        raise_error(a.err, kErrInvalid);
        U.u = n_units;
      } else {
        U.k0 = U.split * split_keys;
        U.k1 = min(ctx, U.k0 + split_keys);
      }
    }
    slot = U;
  };
  auto load_q_raw = [&](const Unit& U, uint4 (&q)[GU]) {
#pragma unroll
    for (int hh = 0; hh < GU; ++hh)
      q[hh] = *reinterpret_cast<const uint4*>(static_cast<const T*>(a.q) + (size_t(U.t) * H + U.h0 + hh) * A +
                                              c * EPV);
  };
  // tiles of unit U that this warp takes (tiles warp, warp + kWarps, ...)
  auto warp_tiles = [&](const Unit& U) -> int {
    if (U.u >= n_units) return 0;
    const int nt = (U.k1 - U.k0 + kTile - 1) / kTile;
    return nt > warp ? (nt - warp + kWarps - 1) / kWarps : 0;
  };
  uint32_t issued = 0, consumed = 0;        // this warp's ring positions (warp-uniform)
  // lane 0 copies the warp's o-th tile of unit U into the next ring slot
  auto issue = [&](const Unit& U, int o) {
    if (lane == 0) {
      const int j0 = U.k0 + (warp + kWarps * o) * kTile;
      const int st = issued % kStages;
      const uint32_t bar = sm100::smem_u32(&bars[st]);
      const int blk = a.block_tables[size_t(U.s) * a.max_blocks_per_seq + j0 / B];
      if (blk >= 0 && blk < a.num_blocks) {
        valid[st] = 1;
        const size_t off = size_t(blk) * blk_stride + size_t(U.hkv) * B * A + size_t(j0 % B) * A;
        const uint32_t dst = sm100::smem_u32(ring + st * 2 * kTileBytes);
        sm100::mbar_arrive_expect_tx(bar, 2 * kTileBytes);
        sm100::bulk_load(dst, kp + off, kTileBytes, bar);
        sm100::bulk_load(dst + kTileBytes, vp + off, kTileBytes, bar);
      } else {
        raise_error(a.err, kErrBounds);
        valid[st] = 0;
        sm100::mbar_arrive(bar);
      }
    }
    ++issued;
  };

  // Units are claimed two ahead: unit j lives in slot j % 2.  While unit k
  // runs, unit k + 1 is known (its first tiles are already being copied) and
  // one thread claims unit k + 2, so the claim's round trips to L2 hide
  // behind the tile stream; the claiming thread rotates over the warps.
  if (threadIdx.x == 0) {
    claim(slots[0]);
    claim(slots[1]);
  }
  __syncthreads();
  Unit U0 = slots[0];
  int n0 = warp_tiles(U0), i0 = 0;          // tiles of U0: count, issued so far
  uint4 q_raw[GU];                          // this lane's 16 bytes of U0's query rows
#pragma unroll
  for (int hh = 0; hh < GU; ++hh) q_raw[hh] = make_uint4(0, 0, 0, 0);
  if (U0.u < n_units) load_q_raw(U0, q_raw);
  for (int k = 0; U0.u < n_units; ++k) {
    __syncthreads();                        // slot (k + 1) % 2 written; slot k % 2 read by every thread
    const Unit U1 = slots[(k + 1) & 1];
    if (threadIdx.x == (k % kWarps) * 32) claim(slots[k & 1]);
    const int n1 = warp_tiles(U1);
    int i1 = 0;
    auto top_up = [&]() {
      while (issued - consumed < uint32_t(kStages)) {
        if (i0 < n0)
          issue(U0, i0++);
        else if (i1 < n1)
          issue(U1, i1++);
        else
          break;
      }
    };
    top_up();
    float qf[GU][EPV];
#pragma unroll
    for (int hh = 0; hh < GU; ++hh) {
      Vec16<T>::to_float(q_raw[hh], qf[hh]);
#pragma unroll
      for (int e = 0; e < EPV; ++e) qf[hh][e] *= a.scale_log2;    // scores in the exp2 domain
    }
    if (U1.u < n_units) load_q_raw(U1, q_raw);                   // in flight while U0 streams
    float m_run[GU], l_run[GU];
    float acc[GU][EPV];
#pragma unroll
    for (int hh = 0; hh < GU; ++hh) {
      m_run[hh] = -INFINITY;
      l_run[hh] = 0.f;
#pragma unroll
      for (int e = 0; e < EPV; ++e) acc[hh][e] = 0.f;
    }
    for (int it = 0; it < n0; ++it) {
      const int st = consumed % kStages;
      if (!__all_sync(0xffffffffu, sm100::mbar_wait(sm100::smem_u32(&bars[st]), (consumed / kStages) & 1))) {
        if (lane == 0) {
          raise_error(a.err, kErrTimeout | kSiteDecodeRing);
          abort_flag = 1;
        }
        break;
      }
      const int base = U0.k0 + (warp + kWarps * it) * kTile;
      const bool ok = valid[st] != 0;
      const uint8_t* kt = ring + st * 2 * kTileBytes;
      uint4 kv[NR], vv[NR];
#pragma unroll
      for (int i = 0; i < NR; ++i) {
        const int r = g + RPL * i;
        const bool in = ok && base + r < U0.k1;
        kv[i] = in ? *reinterpret_cast<const uint4*>(kt + r * 256 + c * 16) : make_uint4(0, 0, 0, 0);
        vv[i] = in ? *reinterpret_cast<const uint4*>(kt + kTileBytes + r * 256 + c * 16) : make_uint4(0, 0, 0, 0);
      }
      if (GU == 1)
        tile_update<T, EPV, LPR, RPL, NR>(qf[0], kv, vv, base, U0.k1, lane, m_run[0], l_run[0], acc[0]);
      else
        group_tile_update<GU, EPV, LPR, RPL, NR>(qf, kv, vv, base, U0.k1, lane, m_run, l_run, acc);
      __syncwarp();                         // every lane has used what it read: the slot may be refilled
      ++consumed;
      top_up();
    }
    if (GU > 1) {                           // the grouped update keeps per-lane row sums
#pragma unroll
      for (int hh = 0; hh < GU; ++hh) l_run[hh] = warp_sum(l_run[hh]);
    }
    finish_group<GU>(sa, U0, m_run, l_run, acc, sm);
    U0 = U1;
    n0 = n1;
    i0 = i1;
  }
  // after a timeout some copies may still be in flight: wait for them (bounded) before exiting
  while (consumed < issued) {
    sm100::mbar_wait(sm100::smem_u32(&bars[consumed % kStages]), (consumed / kStages) & 1);
    ++consumed;
  }
  __syncthreads();                          // every claim of this CTA has returned
  if (threadIdx.x == 0) release_claims(sa.claims, sa.done, min(int(gridDim.x), n_units));
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

size_t split_kv_workspace_bytes(bool row_mode, int32_t num_seqs, int32_t num_tokens,
                                int32_t num_heads, int32_t head_dim, int32_t max_context_len) {
  if (!row_mode) return step_workspace_bytes(num_seqs, num_tokens, num_heads, head_dim, max_context_len);
  const size_t rows = size_t(num_tokens);
  const size_t splits = size_t((max_context_len + kSplitKeys - 1) / kSplitKeys);
  if (rows == 0 || splits <= 1) return 256;
  return align256(rows * num_heads * sizeof(int32_t)) +
         rows * num_heads * splits * (head_dim + 2) * sizeof(float);
}

template <typename T, int A, bool ROW>
static void launch(const SplitArgs& sa, dim3 grid, cudaStream_t stream) {
  split_kv_kernel<T, A, ROW><<<grid, kWarps * 32, 0, stream>>>(sa);
}

// Query heads per decode unit: all G query heads of a key/value head on the
// tensor-core path; otherwise the largest of 4, 3, 2, 1 dividing G (1 for
// multi-head attention).
int decode_group_heads(const AttnArgs& a) {
  const int G = a.num_kv_heads > 0 ? a.num_heads / a.num_kv_heads : 1;
  if (decode_tc_applies(a)) return G;
  for (int gu = 4; gu > 1; --gu)
    if (G % gu == 0) return gu;
  return 1;
}

float decode_rate_for(const AttnArgs& a) {
  if (decode_tc_applies(a)) return decode_tc_rate_per_sm(decode_group_heads(a));
  return decode_rate_per_sm(decode_group_heads(a));
}

float decode_rate_per_sm(int group_heads) {
  switch (group_heads) {
    case 1: return 9.0e4f;
    case 2: return 6.0e4f;
    case 3: return 4.2e4f;
    default: return 3.2e4f;
  }
}

template <int GU>
static int persistent_ctas(int dev) {
  // One-time, per-device set-up; first calls may come from several host
  // threads at once, so it runs under a lock.
  static std::mutex mu;
  static int ctas_per_sm[64] = {};
  static bool ready[64] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (!ready[dev]) {
    cudaError_t e = cudaFuncSetAttribute(split_kv_persistent_kernel<GU>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(bulk_smem_bytes<GU>()));
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&ctas_per_sm[dev], split_kv_persistent_kernel<GU>,
                                                        kWarps * 32, bulk_smem_bytes<GU>());
    if (e != cudaSuccess) {
      cuda_fail(e, "split-KV: kernel attributes");
      return 0;
    }
    if (ctas_per_sm[dev] < 1) ctas_per_sm[dev] = 1;
    ready[dev] = true;
  }
  return ctas_per_sm[dev] * sm_count();
}

void set_decode_plan(const AttnArgs& a, StepPlan* plan) {
  const bool tc = decode_tc_applies(a);
  plan->dec_ctas = decode_persistent_ctas(a);
  plan->dec_groups = a.num_heads / decode_group_heads(a);
  const bool wide = tc && decode_group_heads(a) > 16;
  plan->dec_units_per_cta[0] = wide ? kTcUnitsPerCtaWide : tc ? kTcUnitsPerCta[0] : kUnitsPerCta[0];
  plan->dec_units_per_cta[1] = wide ? kTcUnitsPerCtaWide : tc ? kTcUnitsPerCta[1] : kUnitsPerCta[1];
  plan->kv_bytes_per_key = 2 * a.num_kv_heads * a.head_dim * (a.dtype == CB_DTYPE_BF16 ? 2 : 4);
  plan->dec_bytes_per_us_per_sm = decode_rate_for(a);
}

int decode_persistent_ctas(const AttnArgs& a) {
  if (decode_tc_applies(a)) return decode_tc_ctas();
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    fail(CB_ERR_UNSUPPORTED, "decode: no usable current device");
    return 0;
  }
  switch (decode_group_heads(a)) {
    case 4: return persistent_ctas<4>(dev);
    case 3: return persistent_ctas<3>(dev);
    case 2: return persistent_ctas<2>(dev);
    default: return persistent_ctas<1>(dev);
  }
}

static bool persistent_ok(const AttnArgs& a) {
  return a.dtype == CB_DTYPE_BF16 && a.head_dim == 128 && a.block_size % kTile == 0;
}

cb_status launch_decode_persistent(const AttnArgs& a, const StepPlan& plan, bool after_plan,
                                   bool wait_previous, cudaStream_t stream) {
  NvtxRange nvtx("cb.decode");
  if (decode_tc_applies(a)) return launch_decode_tc(a, plan, after_plan, wait_previous, stream);
  SplitArgs sa;
  sa.wait_previous = wait_previous ? 1 : 0;
  sa.a = a;
  sa.tickets = plan.tickets;
  sa.partials = plan.partials;
  sa.max_splits = plan.max_splits;
  sa.items = plan.dec_items;
  sa.header = plan.header;
  sa.claims = plan.header + 2;
  sa.done = plan.header + 11;
  sa.item_cap = plan.dec_cap;
  sa.tag = plan.tag;
  if (!persistent_ok(a)) {
    // other shapes: one CTA per (split, head, sequence); the plan has cleared the tickets
    if (a.num_kv_heads != a.num_heads)
      return fail(CB_ERR_UNSUPPORTED, "split-KV path: grouped KV heads need bf16, head_dim 128, block size % 16 == 0");
    if (a.num_seqs > 65535) return fail(CB_ERR_UNSUPPORTED, "split-KV path: more than 65535 rows");
    const dim3 grid(unsigned(sa.max_splits), unsigned(a.num_heads), unsigned(a.num_seqs));
    const bool bf16 = a.dtype == CB_DTYPE_BF16;
    if (bf16 && a.head_dim == 128) launch<__nv_bfloat16, 128, false>(sa, grid, stream);
    else if (bf16 && a.head_dim == 64) launch<__nv_bfloat16, 64, false>(sa, grid, stream);
    else if (!bf16 && a.head_dim == 128) launch<float, 128, false>(sa, grid, stream);
    else if (!bf16 && a.head_dim == 64) launch<float, 64, false>(sa, grid, stream);
    else return fail(CB_ERR_UNSUPPORTED, "split-KV path: head_dim must be 64 or 128");
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? CB_OK : cuda_fail(e, "split-KV launch");
  }
  const int gu = decode_group_heads(a);
  sa.n_groups = a.num_heads / gu;
  const int ctas = decode_persistent_ctas(a);
  if (ctas < 1) return CB_ERR_CUDA;
  // never more CTAs than units could exist
  const int64_t max_units = int64_t(a.num_seqs) * plan.max_splits * sa.n_groups;
  const int64_t grid = std::min<int64_t>(ctas, max_units);
  if (grid < 1) return CB_OK;
  cudaError_t e;
  switch (gu) {
    case 4:
      e = launch_kernel(split_kv_persistent_kernel<4>, dim3(unsigned(grid)), dim3(kWarps * 32), bulk_smem_bytes<4>(),
                        stream, after_plan, sa);
      break;
    case 3:
      e = launch_kernel(split_kv_persistent_kernel<3>, dim3(unsigned(grid)), dim3(kWarps * 32), bulk_smem_bytes<3>(),
                        stream, after_plan, sa);
      break;
    case 2:
      e = launch_kernel(split_kv_persistent_kernel<2>, dim3(unsigned(grid)), dim3(kWarps * 32), bulk_smem_bytes<2>(),
                        stream, after_plan, sa);
      break;
    default:
      e = launch_kernel(split_kv_persistent_kernel<1>, dim3(unsigned(grid)), dim3(kWarps * 32), bulk_smem_bytes<1>(),
                        stream, after_plan, sa);
  }
  return e == cudaSuccess ? CB_OK : cuda_fail(e, "split-KV: persistent launch");
}

cb_status launch_split_kv(const AttnArgs& a, bool row_mode, void* workspace,
                          size_t workspace_bytes, cudaStream_t stream) {
  NvtxRange nvtx("cb.decode_rows");
  const int32_t rows = row_mode ? a.num_tokens : a.num_seqs;
  if (rows == 0) return CB_OK;
  if (!row_mode) {
    // decode rows: step plan, then the decode kernel over its items
    StepPlan plan;
    cb_status st = step_plan_layout(workspace, workspace_bytes, a.num_seqs, a.num_tokens, a.num_heads,
                                    a.head_dim, a.max_context_len, &plan);
    if (st != CB_OK) return st;
    set_decode_plan(a, &plan);
    st = launch_plan(a, plan, stream);
    if (st != CB_OK) return st;
    return launch_decode_persistent(a, plan, true, true, stream);
  }
  if (rows > 65535) return fail(CB_ERR_UNSUPPORTED, "split-KV path: more than 65535 rows");
  SplitArgs sa = {};
  sa.a = a;
  sa.max_splits = (a.max_context_len + kSplitKeys - 1) / kSplitKeys;
  const size_t need = split_kv_workspace_bytes(row_mode, a.num_seqs, a.num_tokens, a.num_heads,
                                               a.head_dim, a.max_context_len);
  if (workspace_bytes < need || (need > 256 && !workspace))
    return fail(CB_ERR_INVALID, "workspace too small: %zu bytes given, %zu needed", workspace_bytes, need);
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
    return fail(CB_ERR_INVALID, "workspace must be 256-byte aligned");
  sa.tickets = static_cast<int32_t*>(workspace);
  sa.partials = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                         align256(size_t(rows) * a.num_heads * sizeof(int32_t)));
  if (sa.max_splits > 1) {
    cudaError_t e = cudaMemsetAsync(workspace, 0, size_t(rows) * a.num_heads * sizeof(int32_t), stream);
    if (e != cudaSuccess) return cuda_fail(e, "clearing split tickets");
  }
  const dim3 grid(unsigned(sa.max_splits), unsigned(a.num_heads), unsigned(rows));
  const bool bf16 = a.dtype == CB_DTYPE_BF16;
  if (bf16 && a.head_dim == 128) launch<__nv_bfloat16, 128, true>(sa, grid, stream);
  else if (bf16 && a.head_dim == 64) launch<__nv_bfloat16, 64, true>(sa, grid, stream);
  else if (!bf16 && a.head_dim == 128) launch<float, 128, true>(sa, grid, stream);
  else if (!bf16 && a.head_dim == 64) launch<float, 64, true>(sa, grid, stream);
  else return fail(CB_ERR_UNSUPPORTED, "split-KV path: head_dim must be 64 or 128");
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "split-KV launch");
  return CB_OK;
}

}  // namespace cb
