// cb_selftest_bounded_wait: exercises the bounded mbarrier wait that every
// pipeline wait of the library uses, on a barrier nothing ever arrives at.
#include "device_common.cuh"
#include "runtime.h"
#include "sm100_ptx.cuh"

namespace {

__global__ void bounded_wait_kernel(uint64_t timeout_ns, unsigned* err) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = cb::sm100::smem_u32(&bar);
  if (threadIdx.x == 0) {
    cb::sm100::mbar_init(b, 1);
    cb::sm100::fence_mbar_init();
  }
  __syncthreads();
  // No thread arrives: phase 0 never completes, so the wait must give up.
  const bool ok = cb::sm100::mbar_wait(b, 0, timeout_ns);
  if (!ok && threadIdx.x == 0) cb::raise_error(err, cb::kErrTimeout | cb::kSiteSelfTest);
}

}  // namespace

extern "C" cb_status cb_selftest_bounded_wait(int32_t timeout_ms, void* stream) {
  if (timeout_ms < 1 || timeout_ms > 10000)
    return cb::fail(CB_ERR_INVALID, "cb_selftest_bounded_wait: timeout_ms must be in [1, 10000]");
  unsigned* err = cb::device_error_word();
  if (!err) return CB_ERR_CUDA;
  bounded_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(uint64_t(timeout_ms) * 1000000ull, err);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? CB_OK : cb::cuda_fail(e, "cb_selftest_bounded_wait: launch");
}
