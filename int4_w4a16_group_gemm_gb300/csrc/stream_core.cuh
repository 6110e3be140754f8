// Building blocks of the streaming (CUDA-core) W4A16 kernels.
//
// Work split: a warp owns a slice of K; lane l owns EPL = 8*WPL consecutive
// input columns of that slice (WPL packed words per weight row), holds the
// matching activations of up to MT tokens in registers for the whole
// kernel, and walks over weight rows. A row's packed words come from a
// shared-memory stage (filled by bulk copies), are unpacked in registers and
// multiplied with fp32 FMAs; the per-lane partial is scaled by the group
// scale, and 8 rows at a time are reduced across the warp in a fixed order.
//
// Nibble unpacking without integer->float conversion instructions: nibble j
// of a word sits in bits 4j..4j+3. For the four nibbles of a 16-bit half,
// (half & (0xF << 4c)) | 0x4B000000 is the fp32 number 2^23 + nibble*16^c,
// so subtracting 2^23 + 8*16^c gives (nibble - 8) * 16^c exactly. The
// matching activation is pre-multiplied by 16^-c (an exact power-of-two
// scaling), so each FMA adds the exact product (nibble - 8) * x.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "common.cuh"

namespace w4a16 {

constexpr int kRowsPerChunk = 8;

// Thread budget of a streaming CTA for a token tile of MT: 1024 threads (64
// registers each) for MT <= 2, 512 (128 registers) for MT = 4.
__host__ __device__ constexpr int stream_max_threads(int MT) { return MT == 4 ? 512 : 1024; }

__device__ __forceinline__ float nib_bias(int c) {
  // 2^23 + 8 * 16^c, exact in fp32 for c = 0..3
  return c == 0 ? 8388616.0f : c == 1 ? 8388736.0f : c == 2 ? 8390656.0f : 8421376.0f;
}

__device__ __forceinline__ float nib_prescale(int c) {
  return c == 0 ? 1.0f : c == 1 ? 0.0625f : c == 2 ? 0.00390625f : 0.000244140625f;
}

// Load this lane's EPL activations of token row `xrow` (nullptr -> zeros)
// into xr[], pre-scaled by the nibble-class factor of each column.
template <int EPL, bool BF16>
__device__ __forceinline__ void load_x_slice(const void *xrow, int k0, float (&xr)[EPL]) {
  if (xrow == nullptr) {
#pragma unroll
    for (int i = 0; i < EPL; ++i) xr[i] = 0.f;
    return;
  }
  if constexpr (BF16) {
    const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(xrow) + k0);
#pragma unroll
    for (int v = 0; v < EPL / 8; ++v) {
      const uint4 u = __ldg(src + v);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        xr[v * 8 + 2 * h] = __uint_as_float(w[h] << 16);
        xr[v * 8 + 2 * h + 1] = __uint_as_float(w[h] & 0xFFFF0000u);
      }
    }
  } else {
    const float4 *src = reinterpret_cast<const float4 *>(static_cast<const float *>(xrow) + k0);
#pragma unroll
    for (int v = 0; v < EPL / 4; ++v) {
      const float4 f = __ldg(src + v);
      xr[v * 4 + 0] = f.x;
      xr[v * 4 + 1] = f.y;
      xr[v * 4 + 2] = f.z;
      xr[v * 4 + 3] = f.w;
    }
  }
#pragma unroll
  for (int i = 0; i < EPL; ++i) xr[i] *= nib_prescale((i & 7) & 3);
}

// acc[t] = sum over this lane's EPL columns of (nibble - 8) * x[t], for the
// WPL words in `wd` (word i holds columns 8i .. 8i+7 of the lane's slice).
template <int MT, int WPL>
__device__ __forceinline__ void lane_dot(const uint32_t (&wd)[WPL],
                                         const float (&xr)[MT][8 * WPL], float (&acc)[MT]) {
#pragma unroll
  for (int t = 0; t < MT; ++t) acc[t] = 0.f;
#pragma unroll
  for (int i = 0; i < WPL; ++i) {
    const uint32_t lo = wd[i];
    const uint32_t hi = wd[i] >> 16;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float qlo = __uint_as_float((lo & (0xFu << (4 * c))) | 0x4B000000u) - nib_bias(c);
      const float qhi = __uint_as_float((hi & (0xFu << (4 * c))) | 0x4B000000u) - nib_bias(c);
#pragma unroll
      for (int t = 0; t < MT; ++t) {
        acc[t] = fmaf(qlo, xr[t][8 * i + c], acc[t]);
        acc[t] = fmaf(qhi, xr[t][8 * i + 4 + c], acc[t]);
      }
    }
  }
}

// Reduce part[r][t] (8 rows) over the 32 lanes of the warp, in a fixed
// order. On return every lane holds, in res[t], the full sum of row
// (lane >> 2) & 7.
template <int MT>
__device__ __forceinline__ void warp_reduce_8rows(const float (&part)[kRowsPerChunk][MT],
                                                  float (&res)[MT], int lane) {
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
  float q4[4][MT];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int t = 0; t < MT; ++t) {
      const float send = b4 ? part[i][t] : part[i + 4][t];
      const float keep = b4 ? part[i + 4][t] : part[i][t];
      q4[i][t] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 16);
    }
  float q2[2][MT];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int t = 0; t < MT; ++t) {
      const float send = b3 ? q4[i][t] : q4[i + 2][t];
      const float keep = b3 ? q4[i + 2][t] : q4[i][t];
      q2[i][t] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 8);
    }
#pragma unroll
  for (int t = 0; t < MT; ++t) {
    const float send = b2 ? q2[0][t] : q2[1][t];
    const float keep = b2 ? q2[1][t] : q2[0][t];
    float v = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 4);
    v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
    v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
    res[t] = v;
  }
}

// Load WPL consecutive words from shared memory (16/8/4-byte aligned).
template <int WPL>
__device__ __forceinline__ void load_words(const uint8_t *p, uint32_t (&wd)[WPL]) {
  if constexpr (WPL == 4) {
    const uint4 u = *reinterpret_cast<const uint4 *>(p);
    wd[0] = u.x; wd[1] = u.y; wd[2] = u.z; wd[3] = u.w;
  } else if constexpr (WPL == 2) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    wd[0] = u.x; wd[1] = u.y;
  } else {
    wd[0] = *reinterpret_cast<const uint32_t *>(p);
  }
}

}  // namespace w4a16
