// Device-side helpers shared by the kernels.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "cb.h"

namespace cb {

// Bits of the per-device error word (see cb_check_device_errors).
constexpr unsigned kErrBounds = 1u;
constexpr unsigned kErrTimeout = 2u;
constexpr unsigned kErrInvalid = 4u;

// With kErrTimeout, bits 8 and up name the wait that ran out (one bit per
// site, OR-ed over every CTA that gave up), for the error message.
enum : unsigned {
  kSiteDecodeRing = 1u << 8,
  kSitePfItemFree = 1u << 9,     // prefill K loader: item slot release
  kSitePfKFree = 1u << 10,       // prefill K loader: K stage release
  kSitePfQFree = 1u << 11,       // prefill K loader: Q release
  kSitePfItem = 1u << 12,        // prefill V loader / MMA / softmax: item publication
  kSitePfVFree = 1u << 13,       // prefill V loader: V stage release
  kSitePfVTail = 1u << 14,       // prefill V loader: tail tile landing
  kSitePfQ = 1u << 15,           // prefill MMA: Q landing
  kSitePfK = 1u << 16,           // prefill MMA: K landing
  kSitePfV = 1u << 17,           // prefill MMA: V landing
  kSitePfP = 1u << 18,           // prefill MMA: P written
  kSitePfS = 1u << 19,           // prefill softmax: S ready
  kSitePfO = 1u << 20,           // prefill softmax: P V done
  kSiteSelfTest = 1u << 21,
  kSiteDecodeTc = 1u << 22,      // with a prefill site bit: the same wait in the grouped tensor-core decode
};

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void raise_error(unsigned* word, unsigned bits) {
  atomicOr(word, bits);
}

// A persistent grid's claim counter returns to zero for the next launch over
// the same plan (the layers of a planned step): each CTA that claimed counts
// itself in `done` once it will claim no more, and the last of the
// `claimers` zeroes both.  The next launch reads them only after this grid
// has completed.
__device__ __forceinline__ void release_claims(int32_t* claims, int32_t* done, int claimers) {
  if (atomicAdd(done, 1) == claimers - 1) {
    atomicExch(claims, 0);
    atomicExch(done, 0);
  }
}

// 2^x on the special function unit (PTX ex2.approx; ex2(-inf) = +0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Widen a 16-byte vector of T into fp32 values.
template <typename T>
struct Vec16;

template <>
struct Vec16<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ __forceinline__ static void to_float(const uint4& v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
};

template <>
struct Vec16<float> {
  static constexpr int N = 4;
  __device__ __forceinline__ static void to_float(const uint4& v, float (&f)[4]) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
};

// Round one fp32 value to T (bf16: round to nearest even) and store it.
__device__ __forceinline__ void store1(__nv_bfloat16* dst, float v) { *dst = __float2bfloat16_rn(v); }
__device__ __forceinline__ void store1(float* dst, float v) { *dst = v; }

// Read-only 16-byte global load that bypasses L1 allocation (streamed data).
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

}  // namespace cb
