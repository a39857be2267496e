// shared_prefix_d128.cu -- instantiations of the shared-prefix decode kernel
// for bf16 storage, head_dim 128 (one translation unit per head size so the
// library builds in parallel).
#include "shared_prefix_kernel.cuh"

namespace pkv {

pkv_status launch_shared_prefix_d128(const SpLaunch &L) { return launch_sp_d<__nv_bfloat16, 128>(L); }

}  // namespace pkv
