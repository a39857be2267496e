// shared_prefix_f16_d256.cu -- instantiations of the shared-prefix decode kernel for
// fp16 storage, head_dim 256: one 16-row tile per item (one translation unit
// per type and head size so the library builds in parallel).
#include "shared_prefix_kernel.cuh"

namespace pkv {

pkv_status launch_shared_prefix_f16_d256(const SpLaunch &L) { return launch_sp_d<__half, 256>(L); }

}  // namespace pkv
