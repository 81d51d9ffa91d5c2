// K3: prefill-chunk attention on tcgen05 tensor cores (placeholder).
#include "kernels.h"
#include "runtime.h"

namespace cb {

cb_status launch_prefill_tc(const AttnArgs&, cudaStream_t) {
  return fail(CB_ERR_UNSUPPORTED, "prefill chunks on tensor cores are not built yet");
}

}  // namespace cb
