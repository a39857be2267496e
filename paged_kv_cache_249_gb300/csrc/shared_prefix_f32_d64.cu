// shared_prefix_f32_d64.cu -- shared-prefix decode for fp32 storage, head_dim
// 64 (TF32 tiles; one translation unit per combination so the library
// builds in parallel).
#include "shared_prefix_kernel.cuh"

namespace pkv {

pkv_status launch_shared_prefix_f32_d64(const SpLaunch &L) { return launch_sp_d<float, 64>(L); }

}  // namespace pkv
