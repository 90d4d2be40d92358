// CUDA-core paged attention instantiations: q F16, cache E4M3.
#include "decode_simt.cuh"

namespace pkv {
int launch_simt_f16_e4m3(const AttnParams& p, int head_dim, int g_pad, cudaStream_t s) {
  return launch_simt_typed<F16, E4M3>(p, head_dim, g_pad, s);
}
}  // namespace pkv
