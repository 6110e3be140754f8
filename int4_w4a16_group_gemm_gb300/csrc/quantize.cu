// Per-group symmetric INT4 quantiser on the device (weight preparation).
//
// "The Quiet Commit: How a Single Documentation Edit Marks the Completion of
// a Major Engineering Milestone", section "The INT4 Milestone"
// (quantize_w4a16: symmetric, 8 nibbles per int32 along the input dimension,
// nibble = q + 8, fp32 per-group scales). For each row and group of G
// columns (G = 32, 64 or 128):
//   s = max|w| / 7 (IEEE fp32 division), q = clamp(rint(w / s), -8, 7)
//   (round half to even; q = 0 when s = 0), nibble = q + 8, nibble of
//   column k in bits 4*(k mod 8) of word k/8.
// One warp per group: lane l holds G/32 consecutive columns; the max and
// the packing are warp reductions.
#include <algorithm>

#include "kernels.h"

namespace w4a16 {

namespace {

// One warp per group of 32*C columns; lane l owns columns C*l .. C*l+C-1,
// so a packed word (8 columns) is shared by 8/C lanes.
template <int C>
__global__ void __launch_bounds__(256) quantize_kernel(const float *__restrict__ w, long long groups,
                                                       int32_t *__restrict__ qw,
                                                       float *__restrict__ sc) {
  constexpr int GS = 32 * C;  // group size
  const int lane = threadIdx.x & 31;
  const long long warp0 = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  for (long long gidx = warp0; gidx < groups; gidx += nwarps) {
    float v[C];
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < C; ++j) {
      v[j] = __ldg(w + gidx * GS + lane * C + j);
      amax = fmaxf(amax, fabsf(v[j]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    const float s = __fdiv_rn(amax, 7.0f);
    uint32_t word = 0;
#pragma unroll
    for (int j = 0; j < C; ++j) {
      int q = 0;
      if (s > 0.f) {
        const float r = rintf(__fdiv_rn(v[j], s));
        q = static_cast<int>(fminf(fmaxf(r, -8.0f), 7.0f));
      }
      word |= static_cast<uint32_t>(q + 8) << (4 * ((lane * C + j) & 7));
    }
#pragma unroll
    for (int o = 1; o < 8 / C; o <<= 1) word |= __shfl_xor_sync(0xFFFFFFFFu, word, o);
    if ((lane & (8 / C - 1)) == 0) qw[gidx * (GS / 8) + (lane * C) / 8] = static_cast<int32_t>(word);
    if (lane == 0) sc[gidx] = s;
  }
}

}  // namespace

cudaError_t launch_quantize(const float *w, int N, int K, int group, int32_t *qw, float *sc,
                            cudaStream_t stream) {
  const long long groups = static_cast<long long>(N) * (K / group);
  const DeviceInfo &di = device_info();
  const long long want = (groups + 7) / 8;  // 8 warps per block
  const int grid = static_cast<int>(std::min<long long>(want, static_cast<long long>(di.num_sms) * 16));
  if (group == 32)
    quantize_kernel<1><<<grid, 256, 0, stream>>>(w, groups, qw, sc);
  else if (group == 64)
    quantize_kernel<2><<<grid, 256, 0, stream>>>(w, groups, qw, sc);
  else if (group == 128)
    quantize_kernel<4><<<grid, 256, 0, stream>>>(w, groups, qw, sc);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace w4a16
