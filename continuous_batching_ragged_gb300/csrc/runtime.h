// Per-device runtime state shared by the entry points.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <utility>

#include "host_common.h"

namespace cb {

// Device address of the current device's error word (lazily resolved).
// Returns nullptr and records an error message on failure.
unsigned* device_error_word();

// cuTensorMapEncodeTiled from the driver, fetched through the runtime so the
// library does not link libcuda directly.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled_fn();

// A second stream on the current device plus a fork/join event pair, used to
// run prefill chunks and decode rows of one step concurrently.  The returned
// mutex must be held while the events are recorded and waited on.
struct AuxStream {
  cudaStream_t stream;
  cudaEvent_t fork;
  cudaEvent_t join;
};
AuxStream* aux_stream();
void lock_aux();
void unlock_aux();

// Number of SMs of the current device.
int sm_count();

// A named NVTX range over a host scope (header-only NVTX v3: without an
// attached profiler each push/pop is a cheap no-op).  Marks the launches of
// the append, the step plan, the decode and the prefill kernels, so a
// timeline shows which host call enqueued which kernels.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

cb_status cuda_fail(cudaError_t err, const char* what);

// Launch `kernel` on `stream`.  `after_previous`: programmatic dependent
// launch -- the grid may start while the kernel launched just before it on
// the same stream is still running, and must wait for it on the device
// (griddepcontrol.wait) before reading its results.
template <typename... Params, typename... Args>
cudaError_t launch_kernel(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                          bool after_previous, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = after_previous ? attr : nullptr;
  cfg.numAttrs = after_previous ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace cb
