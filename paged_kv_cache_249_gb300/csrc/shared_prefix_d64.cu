// shared_prefix_d64.cu -- instantiations of the shared-prefix decode kernel
// for bf16 storage, head_dim 64 (one translation unit per head size so the
// library builds in parallel).
#include "shared_prefix_kernel.cuh"

namespace pkv {

pkv_status launch_shared_prefix_d64(const SpLaunch &L) { return launch_sp_d<__nv_bfloat16, 64>(L); }

}  // namespace pkv
