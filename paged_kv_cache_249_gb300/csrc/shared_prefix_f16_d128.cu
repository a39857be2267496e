// shared_prefix_f16_d128.cu -- instantiations of the shared-prefix decode
// kernel for fp16 storage, head_dim 128 (one translation unit per type and
// head size so the library builds in parallel).
#include "shared_prefix_kernel.cuh"

namespace pkv {

pkv_status launch_shared_prefix_f16_d128(const SpLaunch &L) { return launch_sp_d<__half, 128>(L); }

}  // namespace pkv
