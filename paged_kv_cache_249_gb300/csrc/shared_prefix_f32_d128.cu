// shared_prefix_f32_d128.cu -- shared-prefix decode for fp32 storage,
// head_dim 128 (TF32 tiles; one translation unit per combination so the
// library builds in parallel).
#include "shared_prefix_kernel.cuh"

namespace pkv {

pkv_status launch_shared_prefix_f32_d128(const SpLaunch &L) { return launch_sp_d<float, 128>(L); }

}  // namespace pkv
