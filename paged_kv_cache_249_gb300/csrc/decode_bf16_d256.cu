// decode_bf16_d256.cu -- instantiations of the paged decode kernel for
// bf16 storage, head_dim 256 (one translation unit per combination so the
// library builds in parallel).
#include "decode_kernel.cuh"

namespace pkv {

pkv_status launch_decode_bf16_d256(const DecodeLaunch &L) { return launch_d<__nv_bfloat16, 256>(L); }

}  // namespace pkv
