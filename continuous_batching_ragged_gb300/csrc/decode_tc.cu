// K2 for grouped-query heads on tcgen05 tensor cores (bf16, head_dim 128).
//
// Page "continuous-batching" (zhangchitc.github.io), section "Inside the
// kernel": a decoding request's one new query attends every key and value of
// its cache, read block by block and folded into a running state (online
// softmax).  With grouped-query attention (fewer key/value heads than query
// heads; not on the pages) the G query heads that share a key/value head read
// the same K/V stream, so one pass over it can serve all G: their G query rows
// are the A operand of S = Q K^T and P of O += P V, a dense contraction that
// runs on the tensor cores instead of G dot products per key on the FMA pipe.
//
// A unit is (sequence, split, key/value head): the G query rows of one decode
// token against keys [k0, k1) of one split (the step plan's decode items,
// times the key/value heads).  The G rows occupy the first rows of a
// 128-row tile (tcgen05 MMAs have at least 64 rows; the rest are zero), and a
// KV tile is 128 keys of 128/B paged blocks, one 3-D TMA box per block and
// 64-dim half, 128-byte swizzled -- the same boxes as the prefill kernel.
//   * warp 1 (K loader) claims units, publishes them in a two-slot item ring,
//     loads each unit's G query rows (once the previous unit's last S has
//     read the tile) and streams K tiles into a 3-stage ring, looking the
//     block table up four tiles ahead and prefetching those boxes into L2;
//   * warp 2 (V loader) streams V tiles into a 2-stage ring and zeroes the
//     rows past the context in the last paged block (P is 0 there, but
//     0 * NaN is NaN);
//   * warp 3 (MMA, one thread): S into two TMEM buffers in turn, so the
//     scores of tile j+1 are computed while the softmax of tile j runs:
//     S(j) S(j+1) | P(j)V S(j+2) | P(j+1)V S(j+3) ...; S(j+2) overwrites the
//     columns P(j) V reads, which one thread's in-order MMAs keep safe;
//   * warp 0 (softmax and epilogue): lane r owns query row r = TMEM lane r.
//     It masks keys at or past the split's end, keeps the running maximum
//     in the exp2 domain lazily (rescaling O in TMEM, after the previous
//     P V is done, only when the maximum grew by more than 2^8; P V of even
//     and odd tiles complete on two barriers, so that every parity wait on
//     them targets the latest or the current phase), writes P
//     as bf16 over its S columns, and at the unit's end either stores the
//     normalised rows or, for a row cut into splits, its partial (acc, max,
//     sum); the last split of a (sequence, key/value head) to finish merges
//     every split by log-sum-exp.
// One CTA per SM (about 193 KB of shared memory).  Every wait is bounded; a
// timeout sets the device error word and the CTA winds down, freeing TMEM.
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

constexpr int BM = 128;                          // MMA rows: the unit's G query heads, then zeros
constexpr int BN = 128;                          // keys per KV tile
constexpr int HD = 128;                          // head dim
constexpr int kKStages = 3;
constexpr int kVStages = 2;
constexpr int kThreads = 128;
constexpr int kWarpK = 1, kWarpV = 2, kWarpMma = 3;   // warp 0: softmax and epilogue
constexpr int kMaxGroup = 32;                    // query heads per key/value head: one softmax warp
constexpr int kG4CudaCoreUnitsPerSm = 10;        // groups of four go to CUDA cores from this many units per SM
constexpr uint32_t kHalf = BM * 64 * 2;          // one 64-dim swizzled half of a tile: 16 KB
constexpr uint32_t kTile = 2 * kHalf;            // 32 KB
constexpr uint32_t kTmemCols = 512;              // S buffers at 0 and 128, O at 256
constexpr uint32_t kColO = 256;

constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kTile;
constexpr uint32_t kOffV = kOffK + kKStages * kTile;
constexpr uint32_t kOffBar = kOffV + kVStages * kTile;
constexpr int kItemSlots = 2;
constexpr int kItemReaders = 3;                  // V loader, MMA, softmax
enum : int {
  BAR_Q = 0,                   // the unit's query rows landed
  BAR_QE = 1,                  // every S MMA of the unit has read them
  BAR_S = 2,                   // + buffer: S ready
  BAR_P = BAR_S + 2,           // + buffer: P written
  BAR_O = BAR_P + 2,           // + tile parity: one phase per P V of an even / odd tile completed
  BAR_KF = BAR_O + 2,          // + stage: K landed
  BAR_KE = BAR_KF + kKStages,  // + stage: K consumed
  BAR_VF = BAR_KE + kKStages,  // + stage: V landed (tail zeroed)
  BAR_VE = BAR_VF + kVStages,  // + stage: V consumed
  BAR_VTAIL = BAR_VE + kVStages,
  BAR_IF = BAR_VTAIL + 1,      // + slot: work item published
  BAR_IE = BAR_IF + kItemSlots,  // + slot: work item read by every role
  BAR_DONE = BAR_IE + kItemSlots,
  NUM_BARS = BAR_DONE + 1
};
constexpr uint32_t kOffTmemSlot = kOffBar + 8 * NUM_BARS;
constexpr uint32_t kOffItems = kOffTmemSlot + 16;          // kItemSlots items of 48 bytes
constexpr int kLookAhead = 4;
constexpr int kRing = 8;
constexpr uint32_t kOffRing = kOffItems + kItemSlots * 48;  // K and V box rings, kRing x 16 ints each
constexpr uint32_t kSmemBytes = kOffRing + 2 * kRing * 16 * 4 + 1024;
static_assert(kRing > kLookAhead, "ring must outlive the look-ahead");
static_assert(kSmemBytes <= 232448, "shared memory budget");

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void tma_prefetch_l2_3d(const void* tmap, int32_t x, int32_t y, int32_t z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z)
               : "memory");
}

__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// One claimed unit.
struct Item {
  int u;                                           // unit index; >= the unit count: no more work
  int s, g, t, ctx, k0, k1, split, nsplit, j0, nt, pad;
};
static_assert(sizeof(Item) == 48, "item slot");

struct DecodeTcWork {
  const int2* items;        // the plan's decode items (sequence, split), longest first
  const int32_t* header;    // [0] items, [4] call tag, [5] keys per split
  int32_t* claims;          // unit claim counter
  int32_t* done;            // CTAs done claiming (the last resets both)
  int32_t* tickets;         // [num_seqs][kv heads] split arrival counters (zero between calls)
  float* partials;          // [num_seqs][H][max_splits][HD + 2] split results (acc, max, sum)
  int32_t item_cap;
  int32_t max_splits;
  uint32_t tag;
  int32_t wait_previous;
};

// Warp-wide: lane i < 128/B looks up paged block i of KV tile j, stores its
// box index (or an out-of-range index: TMA fills zeros) in the ring slot of
// the unit's jl-th tile, and asks TMA to prefetch that box into L2.
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

__device__ __forceinline__ void load_kv_tile(uint32_t dst, const CUtensorMap* tm, uint32_t bar, int B, const int* zs) {
  const int bpt = BN / B;
  for (int bi = 0; bi < bpt; ++bi) {
    tma_load_3d(dst + bi * B * 128, tm, bar, 0, 0, zs[bi]);
    tma_load_3d(dst + kHalf + bi * B * 128, tm, bar, 64, 0, zs[bi]);
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const AttnArgs a, const DecodeTcWork w) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gsm = smem_raw + (base - raw);
  auto bar = [&](int i) -> uint32_t { return base + kOffBar + 8u * uint32_t(i); };
  Item* items = reinterpret_cast<Item*>(gsm + kOffItems);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int B = a.block_size;
  const int H = a.num_heads;
  const int Hkv = a.num_kv_heads;
  const int G = H / Hkv;

  if (w.wait_previous) grid_dependency_wait();    // the plan kernel has finished
  const uint32_t seen_tag = uint32_t(__ldcg(w.header + 4));
  const int n_items = __ldcg(w.header);
  const int split_keys = __ldcg(w.header + 5);
  if (seen_tag != w.tag || n_items < 0 || n_items > w.item_cap || split_keys < kSplitKeys || split_keys % BN != 0) {
    if (blockIdx.x == 0 && threadIdx.x == 0) raise_error(a.err, kErrInvalid);
    return;
  }
  const int n_units = n_items * Hkv;
  if (int(blockIdx.x) >= n_units) return;

  // rows G..127 of the query tile stay zero for the whole launch
  for (uint32_t o = threadIdx.x * 16; o < kTile; o += kThreads * 16)
    *reinterpret_cast<uint4*>(gsm + kOffQ + o) = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(bar(BAR_Q), 1);
    mbar_init(bar(BAR_QE), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(BAR_S + b), 1);
      mbar_init(bar(BAR_P + b), 1);
    }
    mbar_init(bar(BAR_O), 1);
    mbar_init(bar(BAR_O + 1), 1);
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

  auto read_item = [&](int n, Item& it) -> bool {
    const int slot = n % kItemSlots;
    if (!__all_sync(0xffffffffu, mbar_wait(bar(BAR_IF + slot), (n / kItemSlots) & 1))) return false;
    it = items[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(BAR_IE + slot));
    return true;
  };

  if (warp == kWarpK) {
    // ------------------------------------------------------------ K loader (claims the work)
    int* ring = reinterpret_cast<int*>(gsm + kOffRing);
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
    }
    uint32_t kc = 0;
    int n = 0;
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
        Item it = {};
        it.u = atomicAdd(w.claims, 1);
        if (it.u < n_units) {
          const int2 di = __ldcg(w.items + it.u / Hkv);
          it.g = it.u % Hkv;
          it.s = di.x;
          it.split = di.y;
          bool bad = it.s < 0 || it.s >= a.num_seqs || it.split < 0;
          if (!bad) {
            it.t = __ldcg(a.cu_seqlens_q + it.s);
            it.ctx = __ldcg(a.context_lens + it.s);
            it.nsplit = (it.ctx + split_keys - 1) / split_keys;
            bad = it.t < 0 || it.t >= a.num_tokens || it.ctx < 1 || it.ctx > a.max_context_len ||
                  it.split >= it.nsplit || it.nsplit > w.max_splits;
          }
          if (bad) {                               // never happens with a plan from this call
            raise_error(a.err, kErrInvalid);
            it.u = n_units;
          } else {
            it.k0 = it.split * split_keys;
            it.k1 = min(it.ctx, it.k0 + split_keys);
            it.j0 = it.k0 / BN;
            it.nt = (it.k1 + BN - 1) / BN - it.j0;
          }
        }
        items[slot] = it;
        mbar_arrive(bar(BAR_IF + slot));
      }
      __syncwarp();
      const Item it = items[slot];
      if (it.u >= n_units) break;
      const int32_t* bt = a.block_tables + size_t(it.s) * a.max_blocks_per_seq;
      // the query rows go in once every S MMA of the previous unit has read the old ones
      auto load_q = [&]() -> bool {
        if (n > 0 && !__all_sync(0xffffffffu, mbar_wait(bar(BAR_QE), (n - 1) & 1))) return false;
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(BAR_Q), 2u * uint32_t(G) * 128u);
          tma_load_3d(base + kOffQ, &tm_q, bar(BAR_Q), 0, it.g * G, it.t);
          tma_load_3d(base + kOffQ + kHalf, &tm_q, bar(BAR_Q), 64, it.g * G, it.t);
        }
        __syncwarp();
        return true;
      };
      const int q_at = min(kKStages - 1, it.nt);
      for (int j = 0; j < min(kLookAhead, it.nt); ++j)
        stage_boxes(it.j0 + j, j, B, it.ctx, bt, a, it.g, lane, ring, &tm_k);
      for (int j = 0; j < it.nt; ++j) {
        if (j == q_at && !load_q()) {
          ok = false;
          site = kSitePfQFree;
          break;
        }
        if (j + kLookAhead < it.nt)
          stage_boxes(it.j0 + j + kLookAhead, j + kLookAhead, B, it.ctx, bt, a, it.g, lane, ring, &tm_k);
        const uint32_t gk = kc + j;
        const int st = gk % kKStages;
        if (gk >= kKStages && !__all_sync(0xffffffffu, mbar_wait(bar(BAR_KE + st), ((gk / kKStages) - 1) & 1))) {
          ok = false;
          site = kSitePfKFree;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(BAR_KF + st), kTile);
          load_kv_tile(base + kOffK + st * kTile, &tm_k, bar(BAR_KF + st), B, ring + (j % kRing) * 16);
        }
        __syncwarp();
      }
      if (ok && q_at == it.nt && !load_q()) {
        ok = false;
        site = kSitePfQFree;
      }
      if (!ok) break;
      kc += it.nt;
    }
    if (!ok && lane == 0) raise_error(a.err, kErrTimeout | kSiteDecodeTc | site);
    if (lane == 0) release_claims(w.claims, w.done, min(int(gridDim.x), n_units));
    if (lane == 0) {
      // (error path) let copies still in flight land before the CTA exits
      for (uint32_t gk = kc > uint32_t(kKStages) ? kc - kKStages : 0; gk < kc; ++gk)
        mbar_wait(bar(BAR_KF + gk % kKStages), (gk / kKStages) & 1);
      if (n > 0) mbar_wait(bar(BAR_Q), (n - 1) & 1);
    }
  } else if (warp == kWarpV) {
    // ------------------------------------------------------------ V loader
    int* ring = reinterpret_cast<int*>(gsm + kOffRing) + kRing * 16;
    if (lane == 0) tma_prefetch_desc(&tm_v);
    uint32_t vc = 0, vtail = 0;
    bool ok = true;
    unsigned site = 0;
    for (int n = 0;; ++n) {
      Item it;
      if (!read_item(n, it)) {
        ok = false;
        site = kSitePfItem;
        break;
      }
      if (it.u >= n_units) break;
      const int32_t* bt = a.block_tables + size_t(it.s) * a.max_blocks_per_seq;
      for (int j = 0; j < min(kLookAhead, it.nt); ++j)
        stage_boxes(it.j0 + j, j, B, it.ctx, bt, a, it.g, lane, ring, &tm_v);
      for (int j = 0; j < it.nt; ++j) {
        if (j + kLookAhead < it.nt)
          stage_boxes(it.j0 + j + kLookAhead, j + kLookAhead, B, it.ctx, bt, a, it.g, lane, ring, &tm_v);
        const uint32_t gv = vc + j;
        const int st = gv % kVStages;
        if (gv >= kVStages && !__all_sync(0xffffffffu, mbar_wait(bar(BAR_VE + st), ((gv / kVStages) - 1) & 1))) {
          ok = false;
          site = kSitePfVFree;
          break;
        }
        const int kb = (it.j0 + j) * BN;
        const int r0 = it.ctx - kb;                                // first row past the context
        const int r1 = min(BN, ((it.ctx + B - 1) / B) * B - kb);   // end of the last paged block
        const bool tail = r0 < r1;
        const uint32_t vdst = base + kOffV + st * kTile;
        if (lane == 0) {
          const uint32_t land = tail ? bar(BAR_VTAIL) : bar(BAR_VF + st);
          mbar_arrive_expect_tx(land, kTile);
          load_kv_tile(vdst, &tm_v, land, B, ring + (j % kRing) * 16);
        }
        __syncwarp();
        if (tail) {
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
      vc += it.nt;
    }
    if (!ok && lane == 0) raise_error(a.err, kErrTimeout | kSiteDecodeTc | site);
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA
    Item it;
    uint32_t kc = 0, vc = 0, sc = 0;               // K, V tiles consumed; S buffers used
    bool ok = true;
    unsigned site = 0;
    const uint32_t idS = idesc_bf16_f32(BM, BN, false);    // Q (K-major) x K (K-major)
    const uint32_t idO = idesc_bf16_f32(BM, HD, true);     // P (TMEM) x V (N-contiguous)
    const uint64_t dq = smem_desc(base + kOffQ, 16, 1024);
    const uint64_t dk0 = smem_desc(base + kOffK, 16, 1024);
    const uint64_t dv0 = smem_desc(base + kOffV, kHalf, 1024);
    auto issue_s = [&](uint32_t gk, uint32_t buf) {
      const uint64_t kd = dk0 + (((gk % kKStages) * kTile) >> 4);
#pragma unroll
      for (int k = 0; k < HD / 16; ++k) {
        const uint32_t off16 = ((k / 4) * kHalf + (k % 4) * 32) >> 4;
        mma_f16_ss(tmem + 128 * buf, dq + off16, kd + off16, idS, k > 0);
      }
      mma_commit(bar(BAR_S + buf));
    };
    // global tile i: S(i) and P(i) in buffer i & 1, P(i) V signalled on BAR_O + (i & 1)
    auto issue_pv = [&](uint32_t gv, uint32_t buf, bool accumulate) {
      const uint64_t vd = dv0 + (((gv % kVStages) * kTile) >> 4);
#pragma unroll
      for (int k = 0; k < BN / 16; ++k)
        mma_f16_ts(tmem + kColO, tmem + 128 * buf + k * 8, vd + ((k * 2048) >> 4), idO, accumulate || k > 0);
      mma_commit(bar(BAR_O + buf));
    };
    for (int n = 0; ok; ++n) {
      if (!read_item(n, it)) {
        ok = false;
        site = kSitePfItem;
        break;
      }
      if (it.u >= n_units) break;
      if (lane == 0) {
        if (!mbar_wait(bar(BAR_Q), n & 1)) {
          ok = false;
          site = kSitePfQ;
        }
        // the unit's first one or two S go out at once
        for (int j = 0; ok && j < min(2, it.nt); ++j) {
          if (!mbar_wait(bar(BAR_KF + (kc + j) % kKStages), ((kc + j) / kKStages) & 1)) {
            ok = false;
            site = kSitePfK;
            break;
          }
          tc_fence_after();
          issue_s(kc + j, (sc + j) & 1);
          mma_commit(bar(BAR_KE + (kc + j) % kKStages));
          if (j + 1 == it.nt) mma_commit(bar(BAR_QE));
        }
        // then per tile j: P(j) V, and S(j+2) into the buffer P(j) V has just read
        for (int j = 0; ok && j < it.nt; ++j) {
          const uint32_t gv = vc + j, buf = (sc + j) & 1;
          if (!mbar_wait(bar(BAR_VF + gv % kVStages), (gv / kVStages) & 1)) {
            ok = false;
            site = kSitePfV;
            break;
          }
          if (!mbar_wait(bar(BAR_P + buf), ((sc + j) >> 1) & 1)) {
            ok = false;
            site = kSitePfP;
            break;
          }
          tc_fence_after();
          issue_pv(gv, buf, j > 0);
          mma_commit(bar(BAR_VE + gv % kVStages));
          if (j + 2 < it.nt) {
            const uint32_t gk = kc + j + 2;
            if (!mbar_wait(bar(BAR_KF + gk % kKStages), (gk / kKStages) & 1)) {
              ok = false;
              site = kSitePfK;
              break;
            }
            tc_fence_after();
            issue_s(gk, buf);
            mma_commit(bar(BAR_KE + gk % kKStages));
            if (j + 3 == it.nt) mma_commit(bar(BAR_QE));                    // the unit's last S
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      kc += it.nt;
      vc += it.nt;
      sc += it.nt;
    }
    if (lane == 0) {
      if (!ok) raise_error(a.err, kErrTimeout | kSiteDecodeTc | site);
      mma_commit(bar(BAR_DONE));                   // every MMA issued so far has completed
      mbar_wait(bar(BAR_DONE), 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax and epilogue (warp 0)
    const uint32_t lane_base = tmem + (uint32_t(0) << 16);   // warp 0: TMEM lanes 0-31, lane r = row r
    const float sl2 = a.scale_log2;
    uint32_t sc = 0;                               // tiles done (global tile index of the unit's first)
    bool ok = true;
    unsigned site = 0;
    for (int n = 0; ok; ++n) {
      Item it;
      if (!read_item(n, it)) {
        ok = false;
        site = kSitePfItem;
        break;
      }
      if (it.u >= n_units) break;
      float m = -INFINITY, l = 0.f;
      for (int j = 0; ok && j < it.nt; ++j) {
        const uint32_t buf = (sc + j) & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(bar(BAR_S + buf), ((sc + j) >> 1) & 1))) {
          ok = false;
          site = kSitePfS;
          break;
        }
        tc_fence_after();
        uint32_t sr[128];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(lane_base + 128 * buf + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&sr[32 * c]));
        tmem_wait_ld();
        const int kb = (it.j0 + j) * BN;
        if (kb + BN > it.k1) {                     // keys at or past the split's end
#pragma unroll
          for (int c = 0; c < BN; ++c)
            if (kb + c >= it.k1) sr[c] = __float_as_uint(-INFINITY);
        }
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};   // independent chains
#pragma unroll
        for (int c = 0; c < BN; c += 4)
#pragma unroll
          for (int u = 0; u < 4; ++u) m4[u] = fmaxf(m4[u], __uint_as_float(sr[c + u]));
        const float mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        const float m_new = fmaxf(m, mt * sl2);
        const bool resc = m_new > m + 8.0f;        // keep a stale max while exp2 stays <= 2^8
        const float m_use = resc ? m_new : m;
        const float alpha = resc ? ex2(m - m_new) : 1.0f;
        // a row that sees no key yet (only when every key of the tile is masked) keeps m = -inf
        const float m_sub = m_use == -INFINITY ? 0.f : m_use;
        float rs4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const float p0 = ex2(fmaf(__uint_as_float(sr[2 * c]), sl2, -m_sub));
          const float p1 = ex2(fmaf(__uint_as_float(sr[2 * c + 1]), sl2, -m_sub));
          rs4[c & 3] += p0 + p1;
          sr[c] = pack_bf16x2(p0, p1);
        }
        const float rs = (rs4[0] + rs4[1]) + (rs4[2] + rs4[3]);
        l = l * alpha + rs;
        m = m_use;
        if (j > 0 && __any_sync(0xffffffffu, resc)) {
          // O holds P V of tiles < j: wait for the last of them, then rescale.
          // Tile i - 1's barrier (one phase per other tile) has finished the
          // phase of tile i - 3 (S(i) seen implies P(i-2) V done) and cannot
          // pass the phase of tile i + 1 (its P is not written): the parity
          // wait sees exactly tile i - 1's phase
          const uint32_t i1 = sc + j - 1;
          if (!__all_sync(0xffffffffu, mbar_wait(bar(BAR_O + (i1 & 1)), (i1 >> 1) & 1))) {
            ok = false;
            site = kSitePfO;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t o[32];
            tmem_ld32(lane_base + kColO + 32 * c, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(lane_base + kColO + 32 * c, o);
          }
        }
        tmem_st32(lane_base + 128 * buf, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
        tmem_st32(lane_base + 128 * buf + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BAR_P + buf));
      }
      if (!ok) break;
      // every P V of the unit done: those of its last two tiles (one per
      // barrier; each barrier's earlier phases are done and its next one
      // needs a P of the next unit, so each parity wait sees exactly its tile)
      const uint32_t il = sc + it.nt - 1;
      bool okw = mbar_wait(bar(BAR_O + (il & 1)), (il >> 1) & 1);
      if (it.nt >= 2) okw = okw && mbar_wait(bar(BAR_O + ((il - 1) & 1)), ((il - 1) >> 1) & 1);
      if (!__all_sync(0xffffffffu, okw)) {
        ok = false;
        site = kSitePfO;
        break;
      }
      tc_fence_after();
      const bool real = lane < G;
      const int h = it.g * G + lane;
      if (it.nsplit == 1) {
        const float inv = 1.0f / l;
        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.out) + (size_t(it.t) * H + h) * HD;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld32(lane_base + kColO + 32 * c, o);
          tmem_wait_ld();
          if (real) {
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
        // this split's rows, unnormalised, then a ticket per (sequence, key/value head)
        float* part = w.partials + ((size_t(it.s) * H + h) * w.max_splits + it.split) * (HD + 2);
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld32(lane_base + kColO + 32 * c, o);
          tmem_wait_ld();
          if (real) {
            // a split's record is HD + 2 floats (520 bytes): 8-byte aligned, not 16
            float2* p2 = reinterpret_cast<float2*>(part + 32 * c);
#pragma unroll
            for (int e = 0; e < 16; ++e)
              __stcg(p2 + e, make_float2(__uint_as_float(o[2 * e]), __uint_as_float(o[2 * e + 1])));
          }
        }
        if (real) {
          __stcg(part + HD, m);
          __stcg(part + HD + 1, l);
        }
        __threadfence();
        __syncwarp();
        int last = 0;
        if (lane == 0) {
          int32_t* ticket = w.tickets + size_t(it.s) * Hkv + it.g;
          last = atomicAdd(ticket, 1) == it.nsplit - 1;
          if (last) *ticket = 0;                   // every split is in: ready for the next call
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
          __threadfence();                         // acquire: the other splits' partials are read after this
          if (real) {
            const float* rows = w.partials + (size_t(it.s) * H + h) * w.max_splits * (HD + 2);
            float mx = -INFINITY;
            for (int k = 0; k < it.nsplit; ++k) mx = fmaxf(mx, __ldcg(rows + size_t(k) * (HD + 2) + HD));
            float sum = 0.f;
            for (int k = 0; k < it.nsplit; ++k) {
              const float* pk = rows + size_t(k) * (HD + 2);
              sum = fmaf(__ldcg(pk + HD + 1), ex2(__ldcg(pk + HD) - mx), sum);
            }
            const float inv = 1.0f / sum;
            __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.out) + (size_t(it.t) * H + h) * HD;
#pragma unroll 1
            for (int c = 0; c < HD; c += 8) {
              float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
              for (int k = 0; k < it.nsplit; ++k) {
                const float* pk = rows + size_t(k) * (HD + 2);
                const float wk = ex2(__ldcg(pk + HD) - mx) * inv;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const float2 x = __ldcg(reinterpret_cast<const float2*>(pk + c + 2 * e));
                  acc[2 * e] = fmaf(wk, x.x, acc[2 * e]);
                  acc[2 * e + 1] = fmaf(wk, x.y, acc[2 * e + 1]);
                }
              }
              *reinterpret_cast<uint4*>(dst + c) =
                  make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                             pack_bf16x2(acc[6], acc[7]));
            }
          }
        }
      }
      tc_fence_before();                           // O read before the next unit's first P V overwrites it
      sc += it.nt;
    }
    if (!ok && lane == 0) raise_error(a.err, kErrTimeout | kSiteDecodeTc | site);
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
bool g_attr_set[64] = {};

}  // namespace

// Groups of more than four query heads: the CUDA-core kernel's units cover
// at most four, so it would stream each K/V tile G/4 times (or G times for a
// G with no divisor in 2..4); here every tile is streamed once for all G.
// Groups of four read the same bytes in both kernels: the choice below is by
// measured time.  Groups of two and three keep the CUDA-core kernel.
bool decode_tc_applies(const AttnArgs& a) {
  const int G = a.num_kv_heads > 0 ? a.num_heads / a.num_kv_heads : 1;
  const int B = a.block_size;
  if (!(a.dtype == CB_DTYPE_BF16 && a.head_dim == HD && G >= 4 && G <= kMaxGroup &&
        a.num_heads == G * a.num_kv_heads && B >= 16 && B <= BN && (B & (B - 1)) == 0))
    return false;
  if (G > 4) return true;
  // Groups of four: the CUDA-core kernel is faster on large decode-only
  // steps, this one elsewhere.  Measured on GB300 at 32/8 heads (CUDA cores
  // against tensor cores): decode steps of 256 rows 0.446 / 0.469 ms, 200
  // rows 0.378 / 0.378, 160 rows 0.330 / 0.315, 96 rows 0.249 / 0.196;
  // the 2048-token mixed step 0.239 / 0.217; the 32-layer serving trace
  // replayed as CUDA graphs 4.67 / 4.06 ms per step.  Sizes that live on
  // the device (graph replay) take this kernel.
  return a.dims != nullptr || a.max_q_len > 1 ||
         int64_t(a.num_seqs) * a.num_kv_heads < int64_t(kG4CudaCoreUnitsPerSm) * sm_count();
}

// K/V bytes one SM streams per microsecond (measured on GB300, 256-sequence
// decode step: 27 GB/s per SM at G = 8, 14 at G = 32; the unit boundaries,
// one query-row load and one pipeline refill each, bound it, not HBM).
float decode_tc_rate_per_sm(int group_heads) {
  if (group_heads <= 8) return 2.7e4f;
  if (group_heads <= 16) return 2.0e4f;
  return 1.4e4f;
}

int decode_tc_ctas() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(g_attr_mutex);
  if (!g_attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(kSmemBytes));
    if (e != cudaSuccess) {
      cuda_fail(e, "grouped decode: shared memory attribute");
      return 0;
    }
    g_attr_set[dev] = true;
  }
  return sm_count();
}

cb_status launch_decode_tc(const AttnArgs& a, const StepPlan& plan, bool after_previous, bool wait_previous,
                           cudaStream_t stream) {
  NvtxRange nvtx("cb.decode_tc");
  if (!decode_tc_applies(a)) return fail(CB_ERR_UNSUPPORTED, "grouped decode: shape not supported");
  if (int64_t(a.num_blocks) * a.num_kv_heads >= (int64_t(1) << 31))
    return fail(CB_ERR_UNSUPPORTED, "grouped decode: num_blocks * num_kv_heads must fit in int32");
  const int G = a.num_heads / a.num_kv_heads;
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return CB_ERR_CUDA;
  CUtensorMap tq, tk, tv;
  const cuuint32_t ones[3] = {1, 1, 1};
  {
    // q as [tokens][heads][128]: a box is the G query heads of one token, one 64-dim half
    const cuuint64_t dims[3] = {cuuint64_t(HD), cuuint64_t(a.num_heads), cuuint64_t(a.num_tokens)};
    const cuuint64_t strides[2] = {cuuint64_t(HD) * 2, cuuint64_t(a.num_heads) * HD * 2};
    const cuuint32_t box[3] = {64, cuuint32_t(G), 1};
    CUresult r = enc(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.q), dims, strides, box, ones,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(CB_ERR_CUDA, "grouped decode: encoding the Q tensor map failed (%d)", int(r));
  }
  {
    const int B = a.block_size;
    const cuuint64_t dims[3] = {cuuint64_t(HD), cuuint64_t(B), cuuint64_t(a.num_blocks) * a.num_kv_heads};
    const cuuint64_t strides[2] = {cuuint64_t(HD) * 2, cuuint64_t(B) * HD * 2};
    const cuuint32_t box[3] = {64, cuuint32_t(B), 1};
    CUresult r = enc(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.k_pool), dims, strides, box, ones,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r == CUDA_SUCCESS)
      r = enc(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.v_pool), dims, strides, box, ones,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(CB_ERR_CUDA, "grouped decode: encoding the KV tensor maps failed (%d)", int(r));
  }
  const int ctas = decode_tc_ctas();
  if (ctas < 1) return CB_ERR_CUDA;
  DecodeTcWork w;
  w.items = plan.dec_items;
  w.header = plan.header;
  w.claims = plan.header + 2;
  w.done = plan.header + 11;
  w.tickets = plan.tickets;
  w.partials = plan.partials;
  w.item_cap = plan.dec_cap;
  w.max_splits = plan.max_splits;
  w.tag = plan.tag;
  w.wait_previous = wait_previous ? 1 : 0;
  const int64_t max_units = int64_t(plan.dec_cap) * a.num_kv_heads;
  const int64_t grid = std::min<int64_t>(ctas, max_units);
  if (grid < 1) return CB_OK;
  cudaError_t e = launch_kernel(decode_tc_kernel, dim3(unsigned(grid)), dim3(kThreads), kSmemBytes, stream,
                                after_previous, tq, tk, tv, a, w);
  return e == cudaSuccess ? CB_OK : cuda_fail(e, "grouped decode: launch");
}

}  // namespace cb
