// CUDA-core paged attention instantiations: q F16, cache F16.
#include "decode_simt.cuh"

namespace pkv {
int launch_simt_f16_f16(const AttnParams& p, int head_dim, int g_pad, cudaStream_t s) {
  return launch_simt_typed<F16, F16>(p, head_dim, g_pad, s);
}
}  // namespace pkv
