// CUDA-core paged attention instantiations: q BF16, cache BF16.
#include "decode_simt.cuh"

namespace pkv {
int launch_simt_bf16_bf16(const AttnParams& p, int head_dim, int g_pad, cudaStream_t s) {
  return launch_simt_typed<BF16, BF16>(p, head_dim, g_pad, s);
}
}  // namespace pkv
