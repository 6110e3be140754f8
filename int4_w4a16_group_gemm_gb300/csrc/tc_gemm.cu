// Large-M W4A16 GEMM on tcgen05 tensor cores (bf16 activations).
#include "kernels.h"

namespace w4a16 {

bool tc_gemm_supported(int, int, int) { return false; }

cudaError_t launch_tc_gemm(const uint16_t *, const int32_t *, const float *, int, int, int,
                           float *, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace w4a16
