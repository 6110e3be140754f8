// MoE block around the grouped expert layer of moe.cu: the router (logits,
// sigmoid gate, top-k, routing weights) and the shared expert's SwiGLU.
//
// "The Quiet Commit: How a Single Documentation Edit Marks the Completion of
// a Major Engineering Milestone", section "The Context: A Native DDTree
// Engine Takes Shape", and "The Quiet Commit: How a Single Plan Update
// Closed Phase 3 of a Native DDTree Inference Engine", section "The
// Context: Phase 3 of a Custom Inference Stack": a DeepSeekV3/Kimi-style
// MoE with routing and a shared expert; section "The INT4 Milestone": the
// routed and the shared experts run through the INT4 path. The pages give
// no gate formula; the gate is the published DeepSeek-V3 one:
//   l[t][e] = x[t] . W_r[e]   (fp32 router weights, fp32 accumulation)
//   s = sigmoid(l); the topk experts with the largest s + b (b an optional
//   per-expert selection bias), in decreasing order, equal values to the
//   lower expert id; w_j = scale * s_j / (s_0 + ... + s_{k-1}).
// The shared expert is a SwiGLU expert every token uses with weight 1: its
// gate/up and down projections are plain W4A16 GEMMs (whichever kernel the
// token count selects), the SwiGLU between them is swiglu_kernel below, and
// its output is added after the routed slots by the combine in moe.cu.
#include <climits>

#include "common.cuh"
#include "kernels.h"

namespace w4a16 {

namespace {

// ------------------------------------------------------------ router logits
// A warp owns a tile of kRtTok tokens x kRtExp experts; lane l covers the
// columns k = 128 i + 4 l .. 4 l + 3, reading x and W_r as 16-byte vectors
// straight from global memory (both stay in L2: x is [T][H], W_r [E][H]).
// The lane sums its columns in order, then the 32 lane partials of each
// output are added in lane order through shared memory.
constexpr int kRtTok = 8;
constexpr int kRtExp = 8;
constexpr int kRtWarps = 4;

template <bool BF16>
__global__ void __launch_bounds__(32 * kRtWarps)
    router_logits_kernel(const void *__restrict__ x, const float *__restrict__ wr, int T, int H,
                         int E, int tiles_e, int tiles, float *__restrict__ logits, int *status) {
  __shared__ float red[kRtWarps][kRtTok * kRtExp][33];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x * kRtWarps + warp;
  if (tile >= tiles) return;  // no block-wide barrier follows
  const int t0 = (tile / tiles_e) * kRtTok, e0 = (tile % tiles_e) * kRtExp;
  // rows past T or E read the last valid row and are never stored
  size_t xoff[kRtTok], woff[kRtExp];
#pragma unroll
  for (int t = 0; t < kRtTok; ++t) xoff[t] = static_cast<size_t>(min(t0 + t, T - 1)) * H;
#pragma unroll
  for (int e = 0; e < kRtExp; ++e) woff[e] = static_cast<size_t>(min(e0 + e, E - 1)) * H;

  float acc[kRtTok][kRtExp];
#pragma unroll
  for (int t = 0; t < kRtTok; ++t)
#pragma unroll
    for (int e = 0; e < kRtExp; ++e) acc[t][e] = 0.f;

  for (int k = lane * 4; k < H; k += 128) {
    if (!W4A16_IN_BOUNDS(k + 4 <= H, status)) break;  // 4 columns per 16-byte load
    float4 xv[kRtTok];
#pragma unroll
    for (int t = 0; t < kRtTok; ++t) {
      if (BF16) {
        const uint2 r = __ldg(reinterpret_cast<const uint2 *>(
            static_cast<const uint16_t *>(x) + xoff[t] + k));
        xv[t] = make_float4(__uint_as_float(r.x << 16), __uint_as_float(r.x & 0xFFFF0000u),
                            __uint_as_float(r.y << 16), __uint_as_float(r.y & 0xFFFF0000u));
      } else {
        xv[t] = __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(x) + xoff[t] + k));
      }
    }
#pragma unroll
    for (int e = 0; e < kRtExp; ++e) {
      const float4 w = __ldg(reinterpret_cast<const float4 *>(wr + woff[e] + k));
#pragma unroll
      for (int t = 0; t < kRtTok; ++t) {
        float a = acc[t][e];
        a = fmaf(xv[t].x, w.x, a);
        a = fmaf(xv[t].y, w.y, a);
        a = fmaf(xv[t].z, w.z, a);
        a = fmaf(xv[t].w, w.w, a);
        acc[t][e] = a;
      }
    }
  }
#pragma unroll
  for (int t = 0; t < kRtTok; ++t)
#pragma unroll
    for (int e = 0; e < kRtExp; ++e) red[warp][t * kRtExp + e][lane] = acc[t][e];
  __syncwarp();
  for (int i = lane; i < kRtTok * kRtExp; i += 32) {
    float s = 0.f;
    for (int l = 0; l < 32; ++l) s += red[warp][i][l];
    const int t = t0 + i / kRtExp, e = e0 + i % kRtExp;
    if (t < T && e < E) logits[static_cast<size_t>(t) * E + e] = s;
  }
}

// ------------------------------------------------------------ top-k gate
// One warp per token. Lane l holds the scores of experts l, l + 32, ...;
// each of the topk rounds takes the lane-local best untaken expert, then
// the warp-wide best under the order (larger s + b first, then lower id);
// the owner lane marks it taken. Slot j's expert and score end in lane j.
template <int NPL>
__global__ void __launch_bounds__(256)
    router_topk_kernel(const float *__restrict__ logits, const float *__restrict__ bias, int T,
                       int E, int topk, float scale, int32_t *__restrict__ ids,
                       float *__restrict__ route_w, int *status) {
  const int lane = threadIdx.x & 31;
  const int t = static_cast<int>((blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x) >> 5);
  if (t >= T) return;
  float s[NPL], sel[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      s[i] = 1.0f / (1.0f + expf(-logits[static_cast<size_t>(t) * E + e]));
      const float v = s[i] + (bias != nullptr ? bias[e] : 0.0f);
      sel[i] = v == v ? v : -INFINITY;  // a NaN score ranks last
    } else {
      s[i] = 0.f;
      sel[i] = -INFINITY;
    }
  }
  uint32_t taken = 0;
  int my_id = 0;
  float my_s = 0.f, sum = 0.f;
  for (int j = 0; j < topk; ++j) {
    float bv = -INFINITY, bs = 0.f;
    int bi = INT_MAX;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((taken >> i) & 1u) && (sel[i] > bv || (sel[i] == bv && e < bi))) {
        bv = sel[i];
        bi = e;
        bs = s[i];
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
      const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
      const float os = __shfl_xor_sync(0xFFFFFFFFu, bs, o);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
        bs = os;
      }
    }
    // topk <= E, so an untaken expert is always found (bi < E)
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == j) {
      my_id = bi;
      my_s = bs;
    }
    sum += bs;  // the same slot order on every lane
  }
  if (lane < topk && W4A16_IN_BOUNDS(my_id >= 0 && my_id < E, status)) {
    ids[static_cast<size_t>(t) * topk + lane] = my_id;
    route_w[static_cast<size_t>(t) * topk + lane] = scale * my_s / sum;
  }
}

// ------------------------------------------------------------ shared expert SwiGLU
// h[t][i] = silu(gu[t][i]) * gu[t][Is + i], rounded to bf16 when the block
// runs on bf16 activations (the dtype the down projection consumes).
template <bool BF16>
__global__ void swiglu_kernel(const float *__restrict__ gu, int T, int Is, void *__restrict__ h) {
  const size_t n = static_cast<size_t>(T) * Is;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t t = i / Is, c = i % Is;
    const float v = silu_f(gu[t * 2 * Is + c]) * gu[t * 2 * Is + Is + c];
    if (BF16)
      static_cast<__nv_bfloat16 *>(h)[i] = __float2bfloat16_rn(v);
    else
      static_cast<float *>(h)[i] = v;
  }
}

template <int NPL>
cudaError_t launch_topk(const float *logits, const float *bias, int T, int E, int topk,
                        float scale, int32_t *ids, float *route_w, cudaStream_t stream) {
  router_topk_kernel<NPL><<<(T + 7) / 8, 256, 0, stream>>>(logits, bias, T, E, topk, scale, ids,
                                                          route_w, device_info().status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_router(const void *x, bool x_bf16, int T, int H, const float *router_w,
                          const float *bias, int E, int topk, float scale, float *logits,
                          int32_t *ids, float *route_w, cudaStream_t stream) {
  const int tiles_e = (E + kRtExp - 1) / kRtExp;
  const int tiles = ((T + kRtTok - 1) / kRtTok) * tiles_e;
  const int grid = (tiles + kRtWarps - 1) / kRtWarps;
  if (x_bf16)
    router_logits_kernel<true><<<grid, 32 * kRtWarps, 0, stream>>>(x, router_w, T, H, E, tiles_e,
                                                                   tiles, logits, device_info().status);
  else
    router_logits_kernel<false><<<grid, 32 * kRtWarps, 0, stream>>>(x, router_w, T, H, E,
                                                                    tiles_e, tiles, logits,
                                                                    device_info().status);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  if (E <= 128) return launch_topk<4>(logits, bias, T, E, topk, scale, ids, route_w, stream);
  if (E <= 256) return launch_topk<8>(logits, bias, T, E, topk, scale, ids, route_w, stream);
  if (E <= 512) return launch_topk<16>(logits, bias, T, E, topk, scale, ids, route_w, stream);
  return launch_topk<32>(logits, bias, T, E, topk, scale, ids, route_w, stream);
}

cudaError_t launch_swiglu(const float *gu, int T, int Is, bool h_bf16, void *h,
                          cudaStream_t stream) {
  const DeviceInfo &di = device_info();
  const long long n = static_cast<long long>(T) * Is;
  const int grid = static_cast<int>(std::min<long long>((n + 255) / 256, di.num_sms * 8ll));
  if (h_bf16)
    swiglu_kernel<true><<<std::max(grid, 1), 256, 0, stream>>>(gu, T, Is, h);
  else
    swiglu_kernel<false><<<std::max(grid, 1), 256, 0, stream>>>(gu, T, Is, h);
  return cudaGetLastError();
}

}  // namespace w4a16
