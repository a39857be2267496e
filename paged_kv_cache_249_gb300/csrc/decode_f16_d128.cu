// decode_f16_d128.cu -- instantiations of the paged decode kernel for
// fp16 storage, head_dim 128 (one translation unit per combination so the
// library builds in parallel).
#include "decode_kernel.cuh"

namespace pkv {

pkv_status launch_decode_f16_d128(const DecodeLaunch &L) { return launch_d<__half, 128>(L); }

}  // namespace pkv
