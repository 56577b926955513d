// bwd_sm103.cu -- exact attention backward (placeholder until the kernels land).
#include "kernels.h"

namespace attn {

size_t bwd_workspace_bytes(int B, int Hq, int N, int d) {
  const size_t Npad = (size_t)(N + 63) / 64 * 64;
  const size_t rows = (size_t)B * Hq * Npad;
  return (rows * d * 4 + 255) / 256 * 256 + 2 * ((rows * 4 + 255) / 256 * 256);
}

cudaError_t launch_bwd_bf16(int, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                            const CUtensorMap&, const BwdParams&, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace attn
