// shared_prefix_f16_d64.cu -- instantiations of the shared-prefix decode
// kernel for fp16 storage, head_dim 64 (one translation unit per type and
// head size so the library builds in parallel).
#include "shared_prefix_kernel.cuh"

namespace pkv {

pkv_status launch_shared_prefix_f16_d64(const SpLaunch &L) { return launch_sp_d<__half, 64>(L); }

}  // namespace pkv
