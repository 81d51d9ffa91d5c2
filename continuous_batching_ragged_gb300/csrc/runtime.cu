// Library runtime: error reporting, the per-device error word, driver entry
// points and the auxiliary stream.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>

#include "device_common.cuh"
#include "runtime.h"

namespace {

thread_local std::string g_last_error;

// One word per device that loads the library; kernels OR error bits into it.
__device__ unsigned int g_error_word;

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
unsigned* g_error_ptr[kMaxDevices] = {};
cb::AuxStream g_aux[kMaxDevices];
bool g_aux_ready[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};
std::mutex g_aux_mutex;
cb::EncodeTiledFn g_encode = nullptr;

int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}

}  // namespace

namespace cb {

cb_status fail(cb_status status, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return status;
}

cb_status cuda_fail(cudaError_t err, const char* what) {
  return fail(CB_ERR_CUDA, "%s: %s", what, cudaGetErrorString(err));
}

unsigned* device_error_word() {
  int dev = current_device();
  if (dev < 0) {
    fail(CB_ERR_CUDA, "no current CUDA device");
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_error_ptr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_error_word);
    if (e != cudaSuccess) {
      cuda_fail(e, "cudaGetSymbolAddress(error word)");
      return nullptr;
    }
    g_error_ptr[dev] = static_cast<unsigned*>(p);
  }
  return g_error_ptr[dev];
}

EncodeTiledFn encode_tiled_fn() {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
      fail(CB_ERR_CUDA, "cuTensorMapEncodeTiled not available from the driver");
      return nullptr;
    }
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  return g_encode;
}

AuxStream* aux_stream() {
  int dev = current_device();
  if (dev < 0) {
    fail(CB_ERR_CUDA, "no current CUDA device");
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_aux_ready[dev]) {
    AuxStream& a = g_aux[dev];
    cudaError_t e = cudaStreamCreateWithFlags(&a.stream, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&a.fork, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&a.join, cudaEventDisableTiming);
    if (e != cudaSuccess) {
      cuda_fail(e, "creating the auxiliary stream");
      return nullptr;
    }
    g_aux_ready[dev] = true;
  }
  return &g_aux[dev];
}

void lock_aux() { g_aux_mutex.lock(); }
void unlock_aux() { g_aux_mutex.unlock(); }

int sm_count() {
  int dev = current_device();
  if (dev < 0) return 1;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_sms[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    g_sms[dev] = n > 0 ? n : 1;
  }
  return g_sms[dev];
}

}  // namespace cb

extern "C" const char* cb_last_error(void) { return g_last_error.c_str(); }

extern "C" cb_status cb_check_device_errors(void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cb::cuda_fail(e, "cb_check_device_errors: stream synchronize");
  unsigned word = 0;
  e = cudaMemcpyFromSymbol(&word, g_error_word, sizeof(word));
  if (e != cudaSuccess) return cb::cuda_fail(e, "cb_check_device_errors: read error word");
  if (word == 0) return CB_OK;
  const unsigned zero = 0;
  e = cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero));
  if (e != cudaSuccess) return cb::cuda_fail(e, "cb_check_device_errors: clear error word");
  if (word & cb::kErrTimeout)
    return cb::fail(CB_ERR_TIMEOUT, "a bounded device wait ran out (wait sites 0x%x)", word >> 8);
  if (word & cb::kErrBounds) return cb::fail(CB_ERR_BOUNDS, "a slot or block id outside the pool");
  return cb::fail(CB_ERR_INVALID, "device metadata contradicts the host bounds");
}
