// decode_f16_d64.cu -- instantiations of the paged decode kernel for
// fp16 storage, head_dim 64 (one translation unit per combination so the
// library builds in parallel).
#include "decode_kernel.cuh"

namespace pkv {

pkv_status launch_decode_f16_d64(const DecodeLaunch &L) { return launch_d<__half, 64>(L); }

}  // namespace pkv
