// asv_rapid.cu -- RAPID verification kernel (retrieval-augmented target, tail protection,
// adjusted residual sampling).  Placeholder until the kernel lands: the launcher reports
// cudaErrorNotSupported, which the C ABI turns into ASV_ERR_CUDA.
#include "asv_internal.h"

namespace asv {

int rapid_static_smem_bytes() { return 4096; }
int rapid_max_active_clusters(const LaunchPlan&) { return 0; }
cudaError_t launch_rapid(const RapidArgs&, const LaunchPlan&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace asv
