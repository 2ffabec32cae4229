// la_prefill_tc.cu -- tensor-core (tcgen05/TMEM) prefill kernel.  Placeholder until
// the kernel lands: reports every shape as unsupported.
#include "../../include/lightning_attn.h"
#include "la_internal.h"

namespace la {
int prefill_tc_supported(int, int, int64_t) { return LA_ERR_UNSUPPORTED; }
size_t prefill_tc_workspace_bytes(int, int, int64_t) { return 0; }
int launch_prefill_tc(const void*, const void*, const void*, const void*, void*, const float*,
                      float*, float*, int, int, int64_t, float, const Workspace&, cudaStream_t) {
    return LA_ERR_UNSUPPORTED;
}
}  // namespace la
