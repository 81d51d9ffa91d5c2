// K3: prefill-chunk attention on tcgen05 tensor cores (bf16, head_dim 128).
//
// Hugging Face blog "Continuous batching from first principles", section
// "Chunked prefill": a chunk's queries see the keys and values stored for the
// earlier tokens of the prompt plus the chunk's own, with the causal mask
// shifted accordingly; section "Attention": scores Q K^T, mask, row softmax,
// times V.  Page "continuous-batching" (zhangchitc.github.io), section
// "Inside the kernel": the request's cache is read one paged block at a time
// and each block's contribution is accumulated into a running state (online
// softmax).
//
// One CTA computes two 128-row query tiles of one (sequence, head).  Both
// tiles share every K/V tile loaded into shared memory, and the tiles run in
// ping-pong: while one tile's softmax works, the tensor core runs the other
// tile's MMAs.
//   * warp 8 (K loader) and warp 10 (V loader): TMA into a 2-stage K ring and
//     a 3-stage V ring, so a K tile is freed as soon as both S MMAs have read
//     it and the next S never waits behind a V still in use.  Each loader
//     looks up the block table four tiles ahead (one coalesced load per tile
//     into a small shared ring) and asks TMA to prefetch those boxes into L2,
//     so a stage is refilled the moment it frees and the load hits L2.  A 128-key tile
//     is 128/B paged blocks, one 3-D TMA box [B rows x 64 dims] per block and
//     64-dim half, 128-byte swizzled.  Blocks past the context are requested
//     at an out-of-range coordinate, which TMA fills with zeros; the rows of
//     the last, partial block past the context are zeroed by the V loader
//     (P is 0 there but 0 * NaN is NaN).
//   * warp 9 (MMA): one thread issues, per KV tile j, P_0 V_j, S_0(j+1),
//     P_1 V_j, S_1(j+1): S_t = Q_t K^T in fp32 TMEM (K-major SS descriptors),
//     O_t += P_t V with P_t (bf16) read from TMEM and V an N-contiguous B
//     operand.  P_t overwrites the first 64 columns of S_t; S_t(j+1) comes
//     right behind P_t V_j, which the in-order execution of one thread's
//     tcgen05.mma ops keeps safe.  Each tile's softmax thus overlaps the
//     other tile's two MMA groups.
//   * warps 0-3 / 4-7 (softmax of tile 0 / 1): thread i owns query row i =
//     TMEM lane i.  It loads its 128 scores, masks keys j > p + i only on the
//     tiles that cross its warp's diagonal, keeps a running max in the exp2
//     domain (rescaling O in TMEM only when the max grew by more than 2^8),
//     forms exp arguments and row sums two at a time with packed f32x2
//     FMA/add, writes P as bf16 into TMEM, and at the end normalises O and
//     stores its row.
// When a step has few, long query pairs, the plan cuts a pair's key range
// into KV segments that run as separate pieces: each stores its unnormalised
// rows in a partial slot, and the last to finish merges them (log-sum-exp,
// in slot order).
// Every wait is bounded; a timeout sets the device error word and the CTA
// winds down, freeing its TMEM.
#include <algorithm>
#include <mutex>

#include <cuda.h>

#include "device_common.cuh"
#include "kernels.h"
#include "runtime.h"
#include "sm100_ptx.cuh"

namespace cb {
namespace {

using namespace sm100;

constexpr int BM = 128;                          // query rows per tile = TMEM lanes
constexpr int BN = 128;                          // keys per KV tile
constexpr int HD = 128;                          // head dim
constexpr int kQTiles = 2;                       // query tiles per CTA
constexpr int kKStages = 2;                      // K ring depth
constexpr int kVStages = 3;                      // V ring depth (a third V stage beat a third K stage:
                                                 // long-prompt chunk 0.860 against 0.890 ms)
constexpr int kThreads = 352;                    // warps 0-7 softmax, 8 K loader, 9 MMA, 10 V loader
constexpr int kWarpK = 8, kWarpMma = 9, kWarpV = 10;
constexpr uint32_t kHalf = BM * 64 * 2;          // one 64-dim swizzled half: 16 KB
constexpr uint32_t kTile = 2 * kHalf;            // a 128 x 128 bf16 tile: 32 KB
constexpr uint32_t kTmemCols = 512;              // per tile t: S at 256t, O at 256t + 128

constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kQTiles * kTile;
constexpr uint32_t kOffV = kOffK + kKStages * kTile;
constexpr uint32_t kOffBar = kOffV + kVStages * kTile;
constexpr int kItemSlots = 2;                    // claimed work items in flight
constexpr int kItemReaders = 1 + 1 + 8;          // V loader, MMA, softmax warps (one arrival each)
enum : int {
  BAR_Q = 0,                   // Q tiles landed
  BAR_QE = 1,                  // every S MMA of the unit has read Q
  BAR_S = 2,                   // + t: S_t ready
  BAR_P = BAR_S + kQTiles,     // + t: P_t written (128 arrivals)
  BAR_O = BAR_P + kQTiles,     // + t: the piece's last P_t V done
  BAR_KF = BAR_O + kQTiles,    // + stage: K landed
  BAR_KE = BAR_KF + kKStages,  // + stage: K consumed
  BAR_VF = BAR_KE + kKStages,  // + stage: V landed (and its tail zeroed)
  BAR_VE = BAR_VF + kVStages,  // + stage: V consumed
  BAR_VTAIL = BAR_VE + kVStages,
  BAR_IF = BAR_VTAIL + 1,      // + slot: work item published
  BAR_IE = BAR_IF + kItemSlots,  // + slot: work item read by every role
  BAR_DONE = BAR_IE + kItemSlots,  // the MMA thread's last MMAs completed
  NUM_BARS = BAR_DONE + 1
};
constexpr uint32_t kOffTmemSlot = kOffBar + 8 * NUM_BARS;
constexpr uint32_t kOffItems = kOffTmemSlot + 16;  // kItemSlots work items of 48 bytes
constexpr int kLookAhead = 4;                    // tiles of block-table look-ahead and L2 prefetch
constexpr int kRing = 8;                         // box-index ring slots per loader (> kLookAhead)
constexpr uint32_t kOffRing = kOffItems + kItemSlots * 48;  // two rings (K, V) of kRing x 16 ints
constexpr uint32_t kSmemBytes = kOffRing + 2 * kRing * 16 * 4 + 1024;   // + slack to align the base
constexpr int kSlotFloats = (HD + 2) * kPrefillPairRows;   // one partial slot: [HD + 2][256 rows]
static_assert(kRing > kLookAhead, "ring must outlive the look-ahead");
static_assert(kSmemBytes <= 232448, "shared memory budget");

__device__ __forceinline__ void tmem_ld128(uint32_t taddr, uint32_t (&r)[128]) {
#pragma unroll
  for (int c = 0; c < 4; ++c)
    tmem_ld32(taddr + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&r[32 * c]));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Packed fp32 pairs (Blackwell f32x2 FMA / add): two lanes of work per instruction.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ int ld_acquire_gpu(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// The last-arriving segment of a pair merges its warp's rows (this thread:
// `rows`, the row in slot 0) over all nseg segments by log-sum-exp, in slot
// order whoever arrives last, so the bits never depend on timing.  Its own
// segment `mine` comes from TMEM (o_taddr) and registers, the same fp32
// values its partial slot would hold; the others from their slots, two slots
// of 32 dims in flight at a time.  Warp-wide (tcgen05.ld); `store`: this
// thread's row is a real query row.
__device__ __forceinline__ void merge_segments(const float* rows, int nseg, int mine, float m_own, float l_own,
                                               uint32_t o_taddr, __nv_bfloat16* dst, bool store) {
  constexpr int kM = HD * kPrefillPairRows, kL = (HD + 1) * kPrefillPairRows;
  float mx = m_own;
  for (int sg = 0; sg < nseg; ++sg)
    if (sg != mine) mx = fmaxf(mx, __ldcg(rows + size_t(sg) * kSlotFloats + kM));
  float sum = 0.f;
  for (int sg = 0; sg < nseg; ++sg) {
    const float* src = rows + size_t(sg) * kSlotFloats;
    sum += sg == mine ? ex2(m_own - mx) * l_own : ex2(__ldcg(src + kM) - mx) * __ldcg(src + kL);
  }
  const float inv = 1.0f / sum;
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    uint32_t own[32];
    tmem_ld32(o_taddr + 32 * c, own);
    tmem_wait_ld();
    float acc[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) acc[e] = 0.f;
#pragma unroll 1
    for (int sg = 0; sg < nseg; sg += 2) {
      const bool two = sg + 1 < nseg;
      const float* s0 = rows + size_t(sg) * kSlotFloats;
      const float* s1 = s0 + kSlotFloats;
      float v0[32], v1[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        v0[e] = sg == mine ? __uint_as_float(own[e]) : __ldcg(s0 + (32 * c + e) * kPrefillPairRows);
        v1[e] = !two ? 0.f : (sg + 1 == mine ? __uint_as_float(own[e]) : __ldcg(s1 + (32 * c + e) * kPrefillPairRows));
      }
      const float w0 = (sg == mine ? ex2(m_own - mx) : ex2(__ldcg(s0 + kM) - mx)) * inv;
#pragma unroll
      for (int e = 0; e < 32; ++e) acc[e] = fmaf(w0, v0[e], acc[e]);
      if (two) {
        const float w1 = (sg + 1 == mine ? ex2(m_own - mx) : ex2(__ldcg(s1 + kM) - mx)) * inv;
#pragma unroll
        for (int e = 0; e < 32; ++e) acc[e] = fmaf(w1, v1[e], acc[e]);
      }
    }
    if (store) {
      uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * c);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        d4[e] = make_uint4(pack_bf16x2(acc[8 * e], acc[8 * e + 1]), pack_bf16x2(acc[8 * e + 2], acc[8 * e + 3]),
                           pack_bf16x2(acc[8 * e + 4], acc[8 * e + 5]), pack_bf16x2(acc[8 * e + 6], acc[8 * e + 7]));
    }
  }
}

// One KV segment of a segmented pair, after its last P V (warp-wide).  One
// ticket per (pair, query tile, warp): the warp whose segment arrives last
// merges its 32 rows over every segment, so no warp ever waits on another
// warp or CTA.  Every other segment first stores its unnormalised rows (acc,
// max, sum) in its partial slot, dimension-major so a warp's 32 rows are one
// coalesced line.  `rows`: this thread's row in the pair's first slot.
__device__ __forceinline__ void segment_epilogue(float* rows, int32_t* ticket, int nseg, int mine, float m, float l,
                                              uint32_t o_taddr, int lane, __nv_bfloat16* dst, bool store) {
  int merge = 0;
  if (lane == 0 && ld_acquire_gpu(ticket) == nseg - 1) {   // the others are in: no partial needed
    *ticket = 0;                                   // ready for the next call
    merge = 1;
  }
  merge = __shfl_sync(0xffffffffu, merge, 0);
  if (!merge) {
    float* slot = rows + size_t(mine) * kSlotFloats;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t o[32];
      tmem_ld32(o_taddr + 32 * c, o);
      tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 32; ++e) __stcg(slot + (32 * c + e) * kPrefillPairRows, __uint_as_float(o[e]));
    }
    __stcg(slot + HD * kPrefillPairRows, m);
    __stcg(slot + (HD + 1) * kPrefillPairRows, l);
    __threadfence();                               // this row's partial is visible before the ticket
    __syncwarp();
    if (lane == 0 && atomicAdd(ticket, 1) == nseg - 1) {
      *ticket = 0;
      __threadfence();                             // acquire: the other partials are read after this
      merge = 1;
    }
    merge = __shfl_sync(0xffffffffu, merge, 0);
  }
  if (merge) merge_segments(rows, nseg, mine, m, l, o_taddr, dst, store);
}

__device__ __forceinline__ void tma_prefetch_l2_3d(const void* tmap, int32_t x, int32_t y, int32_t z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z)
               : "memory");
}

// Warp-wide: lane i < 128/B looks up paged block i of KV tile j in one coalesced
// load, stores its box index (or `oob`, zero fill) in the ring slot of the
// piece's jl-th tile,
// and asks TMA to prefetch that box into L2 for the load a few tiles later.
__device__ __forceinline__ void stage_boxes(int j, int jl, int B, int ctx, const int32_t* bt, const AttnArgs& a,
                                            int hkv, int lane, int* ring, const CUtensorMap* tm) {
  const int bpt = BN / B;
  if (lane < bpt) {
    const int lb = j * bpt + lane;
    int z = a.num_blocks * a.num_kv_heads;
    if (lb * B < ctx) {
      const int blk = bt[lb];
      if (blk >= 0 && blk < a.num_blocks) {
        z = blk * a.num_kv_heads + hkv;
        tma_prefetch_l2_3d(tm, 0, 0, z);
        tma_prefetch_l2_3d(tm, 64, 0, z);
      } else {
        raise_error(a.err, kErrBounds);
      }
    }
    ring[(jl % kRing) * 16 + lane] = z;
  }
  __syncwarp();
}

__device__ __forceinline__ void load_kv_tile_ring(uint32_t dst, const CUtensorMap* tm, uint32_t bar, int B,
                                                  const int* zs) {
  const int bpt = BN / B;
  for (int bi = 0; bi < bpt; ++bi) {
    tma_load_3d(dst + bi * B * 128, tm, bar, 0, 0, zs[bi]);
    tma_load_3d(dst + kHalf + bi * B * 128, tm, bar, 64, 0, zs[bi]);
  }
}

// One claimed piece of work: KV tiles [j0, j1) of a 256-row query pair of one
// chunk, one head (the whole pair's range unless the plan cut it into
// segments, whose results then go to partial slots slot0 + j0 / segment).
struct WorkItem {
  int u;                                           // entry index; >= the entry count: no more work
  int s, h, row0, c0, q_len, ctx, j0, j1, slot0, pad, spare;   // pad: left-padding rows of the chunk
};
static_assert(sizeof(WorkItem) == 48, "work item slot");

// Shape of a piece: query tiles holding real rows, KV tiles any row of the
// pair can see (the pair's whole range), the piece's first tile and count.
struct UnitShape {
  int nq, p, n_tiles, j0, n;
};
__device__ __forceinline__ UnitShape unit_shape(const WorkItem& it) {
  UnitShape sh;
  sh.nq = it.row0 + BM < it.q_len ? 2 : 1;
  sh.p = it.ctx - it.q_len;                        // cached tokens before this step
  const int kv_end = min(sh.p + it.row0 + sh.nq * BM, it.ctx);
  sh.n_tiles = (kv_end + BN - 1) / BN;
  sh.j0 = it.j0;
  sh.n = it.j1 - it.j0;
  return sh;
}

__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

struct PrefillWork {
  const int4* units;        // the plan's entries (sequence, pair | head << 16, j0 | j1 << 16, slot0)
  int32_t* tickets;         // arrival counters of segmented pairs: [slot0][query tile * 4 + warp]
  float* partials;          // [slot][HD + 2][256 rows] segment results (acc, max, sum), dimension-major
  const int32_t* header;    // [1] = number of units
  int32_t* claims;          // claim counter
  int32_t* done;            // CTAs done claiming (the last resets both)
  int32_t unit_cap;         // capacity of the unit list
  uint32_t tag;             // the plan's call tag
};

// Persistent: a fixed grid of CTAs (one per SM) claims units until none are
// left, in the plan's order: costliest chunk first, head by head, so the
// query pairs of one (sequence, head) run at the same time and share its K/V
// tiles in L2.
// The K loader claims each unit and publishes it in a two-slot ring of work
// items that the V loader, the MMA thread and the softmax warps read in the
// same order; every barrier phase runs on across units, so the next unit's K
// tiles and Q load overlap the end of the current one.
// PADDED: the instantiation for left-padded batches (cb_padded_attention),
// which masks each chunk's pad keys and skips its pad rows' stores; the
// ragged path's instantiation carries none of that code.
template <bool PADDED>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const AttnArgs a, const PrefillWork w) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;    // 128B-swizzled tiles need 1 KB alignment
  uint8_t* gsm = smem_raw + (base - raw);
  auto bar = [&](int i) -> uint32_t { return base + kOffBar + 8u * uint32_t(i); };
  WorkItem* items = reinterpret_cast<WorkItem*>(gsm + kOffItems);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int B = a.block_size;
  const int H = a.num_heads;                       // query heads
  const int G = H / a.num_kv_heads;                // query heads per K/V head (grouped-query attention)

  grid_dependency_wait();                          // the plan kernel has finished
  const uint32_t seen_tag = uint32_t(__ldcg(w.header + 4));
  int n_units = __ldcg(w.header + 1);
  int working = __ldcg(w.header + 8);              // CTAs that take units; the others leave their SM
  const int seg = __ldcg(w.header + 9);            // KV tiles per segment (0: whole pairs)
  if (seen_tag != w.tag || n_units < 0 || n_units > w.unit_cap) {   // a list from another call: no work
    if (blockIdx.x == 0 && threadIdx.x == 0) raise_error(a.err, kErrInvalid);
    n_units = 0;
  }
  // The plan is complete: a decode kernel launched behind this one may start
  // now, on the SMs this grid leaves free.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (working < 1) working = gridDim.x;
  if (int(blockIdx.x) >= min(n_units, working)) return;   // no unit for this CTA: skip the setup

  if (threadIdx.x == 0) {
    mbar_init(bar(BAR_Q), 1);
    mbar_init(bar(BAR_QE), 1);
    for (int t = 0; t < kQTiles; ++t) {
      mbar_init(bar(BAR_S + t), 1);
      mbar_init(bar(BAR_P + t), BM);
      mbar_init(bar(BAR_O + t), 1);
    }
    for (int st = 0; st < kKStages; ++st) {
      mbar_init(bar(BAR_KF + st), 1);
      mbar_init(bar(BAR_KE + st), 1);
    }
    for (int st = 0; st < kVStages; ++st) {
      mbar_init(bar(BAR_VF + st), 1);
      mbar_init(bar(BAR_VE + st), 1);
    }
    mbar_init(bar(BAR_VTAIL), 1);
    for (int i = 0; i < kItemSlots; ++i) {
      mbar_init(bar(BAR_IF + i), 1);
      mbar_init(bar(BAR_IE + i), kItemReaders);
    }
    mbar_init(bar(BAR_DONE), 1);
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(base + kOffTmemSlot, kTmemCols);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gsm + kOffTmemSlot);

  // A reader's view of work item n: wait for it, copy it, release the slot.
  // `arrive`: this thread is its warp's (or role's) one arrival.
  auto read_item = [&](int n, bool arrive, WorkItem& it) -> bool {
    const int slot = n % kItemSlots;
    if (!mbar_wait(bar(BAR_IF + slot), (n / kItemSlots) & 1)) return false;
    it = items[slot];
    if (arrive) mbar_arrive(bar(BAR_IE + slot));
    return true;
  };

  if (warp == kWarpK) {
    // ------------------------------------------------------------ K loader (claims the work)
    int* ring = reinterpret_cast<int*>(gsm + kOffRing);
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
    }
    uint32_t kc = 0;                               // K tiles issued so far
    int n = 0;                                     // units claimed so far
    bool ok = true;
    unsigned site = 0;
    for (;; ++n) {
      const int slot = n % kItemSlots;
      if (n >= kItemSlots &&
          !__all_sync(0xffffffffu, mbar_wait(bar(BAR_IE + slot), ((n / kItemSlots) - 1) & 1))) {
        ok = false;
        site = kSitePfItemFree;
        break;
      }
      if (lane == 0) {
        WorkItem it = {};
        it.u = atomicAdd(w.claims, 1);
        if (it.u < n_units) {
          const int4 pu = __ldcg(w.units + it.u);
          const int qp = pu.y & 0xFFFF;
          it.s = pu.x;
          it.h = pu.y >> 16;
          it.row0 = qp * kPrefillPairRows;
          it.j0 = pu.z & 0xFFFF;
          it.j1 = pu.z >> 16;
          it.slot0 = pu.w;
          bool bad = it.s < 0 || it.s >= a.num_seqs || it.h < 0 || it.h >= H || it.j1 <= it.j0 ||
                     (it.slot0 >= 0 && (seg < 1 || it.slot0 >= kPrefillSegSlots || !w.partials));
          if (!bad) {
            it.c0 = __ldcg(a.cu_seqlens_q + it.s);
            it.q_len = __ldcg(a.cu_seqlens_q + it.s + 1) - it.c0;
            it.ctx = __ldcg(a.context_lens + it.s);
            it.pad = PADDED ? __ldcg(a.pad_lens + it.s) : 0;
            bad = it.c0 < 0 || it.q_len < 2 || it.c0 + it.q_len > a.num_tokens || it.row0 >= it.q_len ||
                  it.ctx < it.q_len || it.ctx > a.max_context_len || it.pad < 0 || it.pad >= it.q_len;
            if (!bad) {
              const UnitShape sh = unit_shape(it);
              bad = it.j1 > sh.n_tiles ||
                    (it.slot0 >= 0 && (it.j0 % seg != 0 || it.j1 != min(it.j0 + seg, sh.n_tiles) ||
                                       sh.n_tiles <= seg ||
                                       it.slot0 + (sh.n_tiles + seg - 1) / seg > kPrefillSegSlots));
            }
          }
          if (bad) {                               // never happens with a plan from this call
            raise_error(a.err, kErrInvalid);
            it.u = n_units;
          }
        }
        items[slot] = it;
        mbar_arrive(bar(BAR_IF + slot));         // release: the slot's contents are visible
      }
      __syncwarp();
      const WorkItem it = items[slot];
      if (it.u >= n_units) break;
      const UnitShape sh = unit_shape(it);
      const int32_t* bt = a.block_tables + size_t(it.s) * a.max_blocks_per_seq;
      // Q of this unit goes in once every S MMA of the previous unit has read
      // the old Q; the first K tiles are requested before that wait.
      auto load_q = [&]() -> bool {
        if (n > 0 && !__all_sync(0xffffffffu, mbar_wait(bar(BAR_QE), (n - 1) & 1))) return false;
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(BAR_Q), kQTiles * kTile);
          for (int t = 0; t < kQTiles; ++t) {
            const int row = it.c0 + it.row0 + t * BM;
            tma_load_3d(base + kOffQ + t * kTile, &tm_q, bar(BAR_Q), 0, it.h, row);
            tma_load_3d(base + kOffQ + t * kTile + kHalf, &tm_q, bar(BAR_Q), 64, it.h, row);
          }
        }
        __syncwarp();
        return true;
      };
      const int q_at = min(kKStages - 1, sh.n);   // K tiles requested before the Q load
      for (int j = 0; j < min(kLookAhead, sh.n); ++j)
        stage_boxes(sh.j0 + j, j, B, it.ctx, bt, a, it.h / G, lane, ring, &tm_k);
      for (int j = 0; j < sh.n; ++j) {
        if (j == q_at && !load_q()) {
          ok = false;
          site = kSitePfQFree;
          break;
        }
        if (j + kLookAhead < sh.n) stage_boxes(sh.j0 + j + kLookAhead, j + kLookAhead, B, it.ctx, bt, a, it.h / G, lane, ring, &tm_k);
        const uint32_t g = kc + j;
        const int st = g % kKStages;
        if (g >= kKStages && !__all_sync(0xffffffffu, mbar_wait(bar(BAR_KE + st), ((g / kKStages) - 1) & 1))) {
          ok = false;
          site = kSitePfKFree;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(BAR_KF + st), kTile);
          load_kv_tile_ring(base + kOffK + st * kTile, &tm_k, bar(BAR_KF + st), B, ring + (j % kRing) * 16);
        }
        __syncwarp();
      }
      if (ok && q_at == sh.n && !load_q()) {
        ok = false;
        site = kSitePfQFree;
      }
      if (!ok) break;
      kc += sh.n;
    }
    if (!ok && lane == 0) raise_error(a.err, kErrTimeout | site);
    if (lane == 0) release_claims(w.claims, w.done, min(int(gridDim.x), min(n_units, working)));
    if (lane == 0) {
      // (error path) let copies still in flight land before the CTA exits
      for (uint32_t g = kc > uint32_t(kKStages) ? kc - kKStages : 0; g < kc; ++g)
        mbar_wait(bar(BAR_KF + g % kKStages), (g / kKStages) & 1);
      if (n > 0) mbar_wait(bar(BAR_Q), (n - 1) & 1);
    }
  } else if (warp == kWarpV) {
    // ------------------------------------------------------------ V loader
    int* ring = reinterpret_cast<int*>(gsm + kOffRing) + kRing * 16;
    if (lane == 0) tma_prefetch_desc(&tm_v);
    uint32_t vc = 0, vtail = 0;                    // V tiles issued, tail fix-ups done
    bool ok = true;
    unsigned site = 0;
    for (int n = 0;; ++n) {
      WorkItem it;
      if (!__all_sync(0xffffffffu, read_item(n, false, it))) {
        ok = false;
        site = kSitePfItem;
        break;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BAR_IE + n % kItemSlots));
      if (it.u >= n_units) break;
      const UnitShape sh = unit_shape(it);
      const int32_t* bt = a.block_tables + size_t(it.s) * a.max_blocks_per_seq;
      for (int j = 0; j < min(kLookAhead, sh.n); ++j)
        stage_boxes(sh.j0 + j, j, B, it.ctx, bt, a, it.h / G, lane, ring, &tm_v);
      for (int j = 0; j < sh.n; ++j) {
        if (j + kLookAhead < sh.n) stage_boxes(sh.j0 + j + kLookAhead, j + kLookAhead, B, it.ctx, bt, a, it.h / G, lane, ring, &tm_v);
        const uint32_t g = vc + j;
        const int st = g % kVStages;
        if (g >= kVStages && !__all_sync(0xffffffffu, mbar_wait(bar(BAR_VE + st), ((g / kVStages) - 1) & 1))) {
          ok = false;
          site = kSitePfVFree;
          break;
        }
        const int kb = (sh.j0 + j) * BN;
        const int r0 = it.ctx - kb;                                // first row past the context
        const int r1 = min(BN, ((it.ctx + B - 1) / B) * B - kb);   // end of the last paged block
        const bool tail = sh.j0 + j == sh.n_tiles - 1 && r0 < r1;
        const uint32_t vdst = base + kOffV + st * kTile;
        if (lane == 0) {
          const uint32_t land = tail ? bar(BAR_VTAIL) : bar(BAR_VF + st);
          mbar_arrive_expect_tx(land, kTile);
          load_kv_tile_ring(vdst, &tm_v, land, B, ring + (j % kRing) * 16);
        }
        __syncwarp();
        if (tail) {
          // zero the stale rows of the last paged block, then publish the tile
          if (!__all_sync(0xffffffffu, mbar_wait(bar(BAR_VTAIL), vtail & 1))) {
            ok = false;
            site = kSitePfVTail;
            break;
          }
          ++vtail;
          uint8_t* vt = gsm + kOffV + st * kTile;
          for (int c = lane; c < (r1 - r0) * 16; c += 32) {
            const int r = r0 + c / 16, wd = c % 16;
            *reinterpret_cast<uint4*>(vt + (wd / 8) * kHalf + r * 128 + (wd % 8) * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(BAR_VF + st));
        }
      }
      if (!ok) break;
      vc += sh.n;
    }
    if (!ok && lane == 0) raise_error(a.err, kErrTimeout | site);
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(BM, BN, false);   // Q (K-major) x K (K-major)
      constexpr uint32_t idO = idesc_bf16_f32(BM, HD, true);    // P (TMEM) x V (N-contiguous)
      // Shared-memory descriptors built once: a descriptor's address field is
      // the byte address / 16 (14 bits, and every address here is below
      // 256 KB), so moving to another tile, stage or K step adds the offset
      // / 16 to the descriptor itself.
      const uint64_t dq0 = smem_desc(base + kOffQ, 16, 1024);
      const uint64_t dk0 = smem_desc(base + kOffK, 16, 1024);
      const uint64_t dv0 = smem_desc(base + kOffV, kHalf, 1024);
      auto issue_s = [&](int t, uint32_t g) {
        const uint64_t kd = dk0 + (((g % kKStages) * kTile) >> 4);
        const uint64_t qd = dq0 + ((t * kTile) >> 4);
#pragma unroll
        for (int k = 0; k < HD / 16; ++k) {
          const uint32_t off16 = ((k / 4) * kHalf + (k % 4) * 32) >> 4;
          mma_f16_ss(tmem + 256 * t, qd + off16, kd + off16, idS, k > 0);
        }
        mma_commit(bar(BAR_S + t));
      };
      // O_t is signalled once per piece, after its last P V: inside a piece
      // the softmax needs no O barrier, because the commit behind S_t(j+1)
      // already covers every earlier MMA of this thread, P_t V_j included.
      auto issue_pv = [&](int t, uint32_t g, bool accumulate, bool last) {
        const uint64_t vd = dv0 + (((g % kVStages) * kTile) >> 4);
#pragma unroll
        for (int k = 0; k < BN / 16; ++k)
          mma_f16_ts(tmem + 256 * t + 128, tmem + 256 * t + k * 8, vd + ((k * 2048) >> 4), idO, accumulate || k > 0);
        if (last) mma_commit(bar(BAR_O + t));
      };
      // Fixed issue order per KV tile j: P_0 V_j, S_0(j+1), P_1 V_j, S_1(j+1).
      // S_t(j+1) overwrites the TMEM columns that P_t V_j reads; tcgen05.mma
      // ops issued by one thread execute in issue order, so the read comes
      // first.  While the softmax of one tile runs, the tensor core works
      // through the other tile's P V and next S.  The first S of the next
      // unit follows the last P V of this one the same way.
      uint32_t kc = 0, vc = 0, cnt0 = 0, cnt1 = 0;  // K, V tiles consumed; S/P/O phases of tiles 0, 1
      bool ok = true;
      unsigned site = 0;
      for (int n = 0; ok; ++n) {
        WorkItem it;
        if (!read_item(n, true, it)) {
          ok = false;
          site = kSitePfItem;
          break;
        }
        if (it.u >= n_units) break;
        const UnitShape sh = unit_shape(it);
        if (!mbar_wait(bar(BAR_Q), n & 1)) {
          ok = false;
          site = kSitePfQ;
          break;
        }
        if (!mbar_wait(bar(BAR_KF + kc % kKStages), (kc / kKStages) & 1)) {
          ok = false;
          site = kSitePfK;
          break;
        }
        tc_fence_after();
        for (int t = 0; t < sh.nq; ++t) issue_s(t, kc);
        mma_commit(bar(BAR_KE + kc % kKStages));
        if (sh.n == 1) mma_commit(bar(BAR_QE));
        for (int j = 0; ok && j < sh.n; ++j) {
          const bool next = j + 1 < sh.n;
          const uint32_t gv = vc + j, gk = kc + j + 1;
          if (!mbar_wait(bar(BAR_VF + gv % kVStages), (gv / kVStages) & 1)) {
            ok = false;
            site = kSitePfV;
            break;
          }
          for (int t = 0; t < sh.nq; ++t) {
            if (!mbar_wait(bar(BAR_P + t), ((t == 0 ? cnt0 : cnt1) + j) & 1)) {
              ok = false;
              site = kSitePfP;
              break;
            }
            tc_fence_after();
            issue_pv(t, gv, j > 0, !next);
            if (t == sh.nq - 1) mma_commit(bar(BAR_VE + gv % kVStages));        // both read V_j
            if (next) {
              if (t == 0 && !mbar_wait(bar(BAR_KF + gk % kKStages), (gk / kKStages) & 1)) {
                ok = false;
                site = kSitePfK;
                break;
              }
              tc_fence_after();
              issue_s(t, gk);
              if (t == sh.nq - 1) {
                mma_commit(bar(BAR_KE + gk % kKStages));                       // both read K_{j+1}
                if (j + 2 == sh.n) mma_commit(bar(BAR_QE));                    // the piece's last S
              }
            }
          }
        }
        kc += sh.n;
        vc += sh.n;
        cnt0 += sh.n;
        if (sh.nq > 1) cnt1 += sh.n;
      }
      if (!ok) raise_error(a.err, kErrTimeout | site);
      mma_commit(bar(BAR_DONE));                   // every MMA issued so far has completed
      mbar_wait(bar(BAR_DONE), 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;                       // query tile of this warpgroup
    const int wq = warp & 3;                       // TMEM lane quarter
    const int i = threadIdx.x - BM * t;            // tile row = TMEM lane
    const uint32_t lane_base = tmem + (uint32_t(wq * 32) << 16) + 256 * t;
    const float sl2 = a.scale_log2;
    uint32_t cnt = 0;                              // S/P phases of this tile consumed
    uint32_t ocnt = 0;                             // O phases (one per piece with rows in this tile)
    bool ok = true;
    unsigned site = 0;
    for (int n = 0; ok; ++n) {
      WorkItem it;
      if (!__all_sync(0xffffffffu, read_item(n, false, it))) {
        ok = false;
        site = kSitePfItem;
        break;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BAR_IE + n % kItemSlots));
      if (it.u >= n_units) break;
      const UnitShape sh = unit_shape(it);
      if (t >= sh.nq) continue;                    // this tile holds no rows of the unit
      const int qi = it.row0 + BM * t + i;         // row within the chunk
      const int limit = min(sh.p + qi, it.ctx - 1);  // last key this row sees
      const int warp_limit = min(sh.p + it.row0 + BM * t + 32 * wq, it.ctx - 1);   // smallest in the warp
      // left padding: keys sh.p .. sh.p + pad - 1 are masked for every row
      const int pad_k0 = sh.p, pad_n = PADDED ? it.pad : 0;
      float m = -INFINITY, l = 0.f;
      for (int j = 0; ok && j < sh.n; ++j) {
        if (!mbar_wait(bar(BAR_S + t), (cnt + j) & 1)) {
          ok = false;
          site = kSitePfS;
          break;
        }
        tc_fence_after();
        uint32_t sr[128];
        tmem_ld128(lane_base, sr);
        tmem_wait_ld();
        const int kb = (sh.j0 + j) * BN;
        float mt = -INFINITY;
        if (kb + BN - 1 > warp_limit) {            // the tile crosses some row's diagonal: mask
#pragma unroll
          for (int c = 0; c < BN; ++c)
            if (kb + c > limit) sr[c] = __float_as_uint(-INFINITY);
        }
        if constexpr (PADDED) {
          if (kb < pad_k0 + pad_n && kb + BN > pad_k0) {   // the tile holds pad keys: mask them
#pragma unroll
            for (int c = 0; c < BN; ++c)
              if (unsigned(kb + c - pad_k0) < unsigned(pad_n)) sr[c] = __float_as_uint(-INFINITY);
          }
        }
        {                                          // four independent max chains (latency, not issue, bound)
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int c = 0; c < BN; c += 8)
#pragma unroll
            for (int u = 0; u < 4; ++u)
              m4[u] = max3(m4[u], __uint_as_float(sr[c + 2 * u]), __uint_as_float(sr[c + 2 * u + 1]));
          mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        }
        const float m_new = fmaxf(m, mt * sl2);
        const bool resc = m_new > m + 8.0f;       // keep a stale max while exp2 stays <= 2^8
        const float m_use = resc ? m_new : m;
        const float alpha = resc ? ex2(m - m_new) : 1.0f;
        const uint64_t scale2 = f2_pack(sl2, sl2);
        // a row that sees no key of the segment so far (a later segment's
        // keys lie past its diagonal) keeps m = -inf and gets p = 0
        const float m_sub = m_use == -INFINITY ? 0.0f : m_use;
        const uint64_t neg_m2 = f2_pack(-m_sub, -m_sub);
        uint64_t sum2[4] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f), f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
        for (int c = 0; c < 64; ++c) {             // P packed in place over the scores
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1])), scale2, neg_m2),
                    x0, x1);
          const float p0 = ex2(x0), p1 = ex2(x1);
          sum2[c & 3] = f2_add(sum2[c & 3], f2_pack(p0, p1));
          sr[c] = pack_bf16x2(p0, p1);
        }
        float rs0, rs1, rs2, rs3, rs4, rs5, rs6, rs7;
        f2_unpack(sum2[0], rs0, rs1);
        f2_unpack(sum2[1], rs2, rs3);
        f2_unpack(sum2[2], rs4, rs5);
        f2_unpack(sum2[3], rs6, rs7);
        const float rs = ((rs0 + rs1) + (rs2 + rs3)) + ((rs4 + rs5) + (rs6 + rs7));
        l = l * alpha + rs;
        m = m_use;
        // S_t(j) done implies P_t V_{j-1} done (one thread issues both, in
        // order, and the commit behind S_t(j) covers all earlier MMAs): O_t
        // is stable for the rescale, and P_t(j) may overwrite P_t(j-1)
        if (j > 0) {
          if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              uint32_t o[32];
              tmem_ld32(lane_base + 128 + 32 * c, o);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
              tmem_st32(lane_base + 128 + 32 * c, o);
            }
          }
        }
        tmem_st32(lane_base, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
        tmem_st32(lane_base + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(BAR_P + t));
      }
      if (!ok) break;
      if (!mbar_wait(bar(BAR_O + t), ocnt & 1)) {
        ok = false;
        site = kSitePfO;
        break;
      }
      tc_fence_after();
      const int e_row = it.c0 + qi, e_h = it.h, e_slot0 = it.slot0, e_j0 = sh.j0, e_ntiles = sh.n_tiles;
      const bool e_real = qi < it.q_len && (!PADDED || qi >= it.pad);   // padding rows are not written
      __nv_bfloat16* const e_dst = static_cast<__nv_bfloat16*>(a.out) + (size_t(e_row) * H + e_h) * HD;
      if (e_slot0 < 0) {
        const float inv = 1.0f / l;
        __nv_bfloat16* dst = e_dst;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld32(lane_base + 128 + 32 * c, o);
          tmem_wait_ld();
          if (e_real) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * c);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float* f = reinterpret_cast<const float*>(&o[8 * e]);
              d4[e] = make_uint4(pack_bf16x2(f[0] * inv, f[1] * inv), pack_bf16x2(f[2] * inv, f[3] * inv),
                                 pack_bf16x2(f[4] * inv, f[5] * inv), pack_bf16x2(f[6] * inv, f[7] * inv));
            }
          }
        }
      } else {
        segment_epilogue(w.partials + size_t(e_slot0) * kSlotFloats + BM * t + i,
                         w.tickets + (e_slot0 * kSegTicketsPerSlot + t * 4 + wq), (e_ntiles + seg - 1) / seg,
                         e_j0 / seg, m, l, lane_base + 128, lane, e_dst, e_real);
      }
      tc_fence_before();                           // O read before the next unit's first P V overwrites it
      cnt += sh.n;
      ++ocnt;
    }
    if (!ok && lane == 0) raise_error(a.err, kErrTimeout | site);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

std::mutex g_attr_mutex;
bool g_attr_set[2][64] = {};

}  // namespace

cb_status launch_prefill_tc(const AttnArgs& a, const StepPlan& plan, bool after_plan, cudaStream_t stream) {
  NvtxRange nvtx("cb.prefill");
  if (a.dtype != CB_DTYPE_BF16 || a.head_dim != HD)
    return fail(CB_ERR_UNSUPPORTED, "prefill chunks: bf16 with head_dim 128 only");
  const int B = a.block_size;
  if (B < 8 || B > BN || (B & (B - 1)) != 0)
    return fail(CB_ERR_UNSUPPORTED, "prefill chunks: block_size must be a power of two in [8, 128]");
  if (int64_t(a.num_blocks) * a.num_kv_heads >= (int64_t(1) << 31))
    return fail(CB_ERR_UNSUPPORTED, "prefill chunks: num_blocks * num_kv_heads must fit in int32");
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return CB_ERR_CUDA;
  CUtensorMap tq, tk, tv;
  const cuuint32_t ones[3] = {1, 1, 1};
  {
    const cuuint64_t dims[3] = {cuuint64_t(HD), cuuint64_t(a.num_heads), cuuint64_t(a.num_tokens)};
    const cuuint64_t strides[2] = {cuuint64_t(HD) * 2, cuuint64_t(a.num_heads) * HD * 2};
    const cuuint32_t box[3] = {64, 1, cuuint32_t(BM)};
    CUresult r = enc(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.q), dims, strides, box,
                     ones, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(CB_ERR_CUDA, "encoding the Q tensor map failed (%d)", int(r));
  }
  {
    const cuuint64_t dims[3] = {cuuint64_t(HD), cuuint64_t(B), cuuint64_t(a.num_blocks) * a.num_kv_heads};
    const cuuint64_t strides[2] = {cuuint64_t(HD) * 2, cuuint64_t(B) * HD * 2};
    const cuuint32_t box[3] = {64, cuuint32_t(B), 1};
    CUresult r = enc(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.k_pool), dims, strides,
                     box, ones, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r == CUDA_SUCCESS)
      r = enc(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.v_pool), dims, strides, box,
              ones, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(CB_ERR_CUDA, "encoding the KV tensor maps failed (%d)", int(r));
  }
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64) {
    std::lock_guard<std::mutex> lock(g_attr_mutex);   // first calls may race from several host threads
    const int v = a.pad_lens ? 1 : 0;
    if (!g_attr_set[v][dev]) {
      cudaError_t e = cudaFuncSetAttribute(v ? prefill_tc_kernel<true> : prefill_tc_kernel<false>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmemBytes));
      if (e != cudaSuccess) return cuda_fail(e, "prefill chunks: shared memory attribute");
      g_attr_set[v][dev] = true;
    }
  }
  PrefillWork w;
  w.units = plan.pre_units;
  w.tickets = plan.pre_tickets;
  w.partials = plan.pre_partials;
  w.header = plan.header;
  w.claims = plan.header + 3;
  w.done = plan.header + 10;
  w.unit_cap = plan.pre_cap * a.num_heads + kPrefillSegSlots;
  w.tag = plan.tag;
  // one CTA per SM, never more than entries could exist
  const int64_t max_units = int64_t(plan.pre_cap) * a.num_heads + kPrefillSegSlots;
  const int64_t grid = std::min<int64_t>(sm_count(), max_units);
  if (grid < 1) return CB_OK;
  cudaError_t e = launch_kernel(a.pad_lens ? prefill_tc_kernel<true> : prefill_tc_kernel<false>,
                                dim3(unsigned(grid)), dim3(kThreads), kSmemBytes, stream, after_plan, tq, tk, tv,
                                a, w);
  if (e != cudaSuccess) return cuda_fail(e, "prefill chunks: launch");
  return CB_OK;
}

}  // namespace cb
