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
// Nibbles are unpacked with the fp16 magic-number trick and mixed-precision
// adds (see nibble_pair in common.cuh): each FMA adds the exact product
// (nibble - 8) * x, with x pre-scaled by 1/16 for the odd nibble classes.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "common.cuh"

namespace w4a16 {

constexpr int kRowsPerChunk = 8;

// Thread budget of a streaming CTA: at most 16 warps, so each thread may
// use 128 registers (8 rows of packed accumulators per token tile plus the
// lane's activations).
__host__ __device__ constexpr int stream_max_threads(int, int = 0) { return 512; }

// Load this lane's EPL activations of token row `xrow` (nullptr -> zeros),
// pre-scaled by the nibble-class factor of each column, as pairs: pair
// 4*i + c of word i holds columns 8i + c and 8i + 4 + c (the two nibbles of
// class c in the word's low and high half).
// Raw activation loads, split from their conversion so that a kernel can
// issue them early and consume them later. fp32: EPL/4 float4; bf16: EPL/8
// uint4 (the uint4 array is sized for the fp32 case).
template <int EPL, bool BF16>
__device__ __forceinline__ void load_x_raw(const void *xrow, int k0, uint4 (&raw)[EPL / 4]) {
  constexpr int NV = BF16 ? EPL / 8 : EPL / 4;
  if (xrow == nullptr) {
#pragma unroll
    for (int v = 0; v < EPL / 4; ++v) raw[v] = make_uint4(0, 0, 0, 0);
    return;
  }
  const uint4 *src = BF16 ? reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(xrow) + k0)
                          : reinterpret_cast<const uint4 *>(static_cast<const float *>(xrow) + k0);
#pragma unroll
  for (int v = 0; v < NV; ++v) raw[v] = __ldg(src + v);
}

// Convert raw activations to the pre-scaled pairs lane_dot consumes: pair
// 4*i + c of word i holds columns 8i + c and 8i + 4 + c (the two nibbles of
// class c in the word's low and high half), times nibble_prescale(c).
template <int EPL, bool BF16>
__device__ __forceinline__ void convert_x(const uint4 (&raw)[EPL / 4], uint64_t (&xp)[EPL / 2]) {
  float xr[EPL];
  if constexpr (BF16) {
#pragma unroll
    for (int v = 0; v < EPL / 8; ++v) {
      const uint32_t w[4] = {raw[v].x, raw[v].y, raw[v].z, raw[v].w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        xr[v * 8 + 2 * h] = __uint_as_float(w[h] << 16);
        xr[v * 8 + 2 * h + 1] = __uint_as_float(w[h] & 0xFFFF0000u);
      }
    }
  } else {
#pragma unroll
    for (int v = 0; v < EPL / 4; ++v) {
      xr[v * 4 + 0] = __uint_as_float(raw[v].x);
      xr[v * 4 + 1] = __uint_as_float(raw[v].y);
      xr[v * 4 + 2] = __uint_as_float(raw[v].z);
      xr[v * 4 + 3] = __uint_as_float(raw[v].w);
    }
  }
#pragma unroll
  for (int i = 0; i < EPL / 8; ++i)
#pragma unroll
    for (int c = 0; c < 4; ++c)
      xp[4 * i + c] = pack_f32x2(xr[8 * i + c] * nibble_prescale(c),
                                 xr[8 * i + 4 + c] * nibble_prescale(c));
}

// Load this lane's EPL activations of token row `xrow` (nullptr -> zeros)
// as pre-scaled pairs (see convert_x).
template <int EPL, bool BF16>
__device__ __forceinline__ void load_x_slice(const void *xrow, int k0, uint64_t (&xp)[EPL / 2]) {
  uint4 raw[EPL / 4];
  load_x_raw<EPL, BF16>(xrow, k0, raw);
  convert_x<EPL, BF16>(raw, xp);
}

// part[r][t] = scale[r] * sum over this lane's columns of (nibble - 8) * x[t]
// for the 8 rows of a stage, with the rows interleaved: for every word and
// nibble class the 8 rows' updates are independent, so 8 FMA chains per
// token are in flight at once. Per word and row: one shift, four logic
// instructions, eight mixed-precision adds and 4 * MT fma.f32x2.
template <int MT, int WPL>
__device__ __forceinline__ void rows_dot(const uint32_t (&wd)[kRowsPerChunk][WPL],
                                         const float (&sv)[kRowsPerChunk],
                                         const uint64_t (&xp)[MT][4 * WPL],
                                         float (&part)[kRowsPerChunk][MT],
                                         const NibbleConsts &k) {
  uint64_t a[kRowsPerChunk][MT];
#pragma unroll
  for (int r = 0; r < kRowsPerChunk; ++r)
#pragma unroll
    for (int t = 0; t < MT; ++t) a[r][t] = 0ull;
#pragma unroll
  for (int i = 0; i < WPL; ++i) {
#pragma unroll
    for (int r = 0; r < kRowsPerChunk; ++r) {
      const uint32_t w = wd[r][i], w8 = w >> 8;
      const uint64_t q[4] = {nibble_pair<0>(w, w8, k), nibble_pair<1>(w, w8, k),
                             nibble_pair<2>(w, w8, k), nibble_pair<3>(w, w8, k)};
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int t = 0; t < MT; ++t) a[r][t] = fma_f32x2(q[c], xp[t][4 * i + c], a[r][t]);
    }
  }
#pragma unroll
  for (int r = 0; r < kRowsPerChunk; ++r)
#pragma unroll
    for (int t = 0; t < MT; ++t) {
      float l, h;
      unpack_f32x2(a[r][t], l, h);
      part[r][t] = (l + h) * sv[r];
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
