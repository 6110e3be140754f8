// Internal host-side launch interface of the W4A16 kernels (not part of the
// public C ABI; the entry points in api.cu validate arguments and call
// these).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/w4a16.h"

namespace w4a16 {

struct DeviceInfo {
  int device = -1;
  int num_sms = 0;
  int smem_optin = 0;  // max dynamic shared memory per block (bytes)
  int *status = nullptr;  // device address of the per-device status word
};

// Per-device facts, looked up once per device (thread-safe).
const DeviceInfo &device_info();

// One-time set-up per device (function attributes such as the dynamic
// shared-memory opt-in are per device): run() calls `fn` once for the
// current device and returns its result on every later call there.
struct PerDeviceOnce {
  static constexpr int kDevices = 64;
  std::once_flag flag[kDevices];
  cudaError_t err[kDevices] = {};
  template <class F>
  cudaError_t run(F &&fn) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevices)
      return cudaErrorInvalidDevice;
    std::call_once(flag[dev], [&] { err[dev] = fn(); });
    return err[dev];
  }
};

// Testing aid: true once after w4a16_debug_fault_next_launch(1); the
// streaming kernel launched then skips its weight copies.
bool take_injected_fault();

// ------------------------------------------------------------ streaming kernel
// y = x * W_hat^T on CUDA cores for any M >= 1 (K % 32 == 0, K <= 16384),
// in one launch: a 2-D grid of row blocks x token tiles of up to 3 tokens.
// `ldx`/`ldy` are row strides in elements. y is fp32, or bf16 (rounded to
// nearest even from the fp32 sum) when `y_bf16`. `overlap` launches with
// programmatic stream serialisation: the weight stream may start before the
// previous kernel on the stream has finished (x and y stay ordered).
cudaError_t launch_stream_gemm(const void *x, bool x_bf16, int ldx, const int32_t *qw,
                               const float *sc, int M, int N, int K, int group, void *y,
                               bool y_bf16, int ldy, bool overlap, cudaStream_t stream);
// Largest K the streaming kernel accepts for a token tile of `mt` (1, 2, 3).
int max_k_stream(int mt);
// Token tile width the streaming kernel uses for M tokens.
int stream_tile(int M, int K);
// Number of streaming-kernel launches for M tokens (1 unless the tiles
// exceed the grid's y limit).
int stream_gemm_passes(int M, int K);

// ------------------------------------------------------------ decode GEMV kernel
// y = x * W_hat^T for one token (M = 1) on CUDA cores, one CTA per SM sized
// so that the next call's CTA can prefetch its weights beside it (see
// gemv.cu). Same `y_bf16` and `overlap` contract as the streaming kernel.
constexpr int kGemvMaxK = 8192;
bool gemv_supported(int M, int N, int K, int group);
cudaError_t launch_gemv(const void *x, bool x_bf16, const int32_t *qw, const float *sc, int N,
                        int K, int group, void *y, bool y_bf16, bool overlap,
                        cudaStream_t stream);

// ------------------------------------------------------------ tensor-core kernel
// Same contract for bf16 activations on tcgen05 tensor cores, including
// `y_bf16` and `overlap`.
cudaError_t launch_tc_gemm(const uint16_t *x, const int32_t *qw, const float *sc, int M,
                           int N, int K, int group, void *y, bool y_bf16, bool overlap,
                           cudaStream_t stream);
bool tc_gemm_supported(int M, int N, int K);
// The small-M form of it (128 weight rows x 64 tokens per tile, K split over
// a cluster of up to `kmax` CTAs, dequantised weights in tensor memory).
cudaError_t launch_tc_split(const uint16_t *x, const int32_t *qw, const float *sc, int M, int N,
                            int K, int group, void *y, bool y_bf16, bool overlap, int kmax,
                            cudaStream_t stream);
// fp32 activations on the tensor cores, exact to fp32 accumulation: each
// activation is split into three bf16 pieces and the group scales are
// applied in fp32 outside the MMA (M <= 64).
cudaError_t launch_tc_f32(const float *x, const int32_t *qw, const float *sc, int M, int N,
                          int K, int group, void *y, bool y_bf16, bool overlap,
                          cudaStream_t stream);
bool tc_f32_supported(int M, int N, int K);

// ------------------------------------------------------------ quantiser
cudaError_t launch_quantize(const float *w, int N, int K, int group, int32_t *qw, float *sc,
                            cudaStream_t stream);

// ------------------------------------------------------------ MoE
cudaError_t launch_moe_sort(const int32_t *ids, int n_pairs, int E, int32_t *offsets,
                            int32_t *perm, cudaStream_t stream);
size_t moe_workspace_bytes(int T, int topk, int E, int H, int I);
// Byte offsets inside that workspace of the expert-sorted pair order, the
// SwiGLU outputs h and the per-slot outputs o.
void moe_workspace_offsets(int T, int topk, int E, int H, int I, size_t *off_perm, size_t *off_h,
                           size_t *off_o);
// `shared_o` ([T][H] fp32, or nullptr) is added to every token's output
// after its routed slots (the shared expert's output).
// Tensor-core expert GEMMs of the MoE layer (moe_tc.cu): bf16 activations,
// n_pairs >= 16, H and I multiples of 256, scale rows whole 16-byte units.
bool moe_tc_supported(int n_pairs, int H, int I, int group);
// xs[s] = x[perm[s] / topk] (bf16 rows of H).
cudaError_t launch_moe_gather(const uint16_t *x, const int32_t *perm, int n, int topk, int H,
                              uint16_t *xs, cudaStream_t stream);
// One expert GEMM over the work items of the sort (token tiles of 16):
// mode 0 gate/up + SwiGLU -> h (bf16, by sorted position) from xs; mode 1
// down x routing weight -> o (fp32, by pair) from h.
cudaError_t launch_moe_tc(int mode, const uint16_t *b, const int32_t *qw, const float *sc,
                          const int32_t *offsets, const int32_t *items, const int32_t *n_items,
                          const int32_t *perm, const float *route_w, int n_pairs, int E, int H,
                          int I, int group, int max_items, void *out, cudaStream_t stream);
cudaError_t launch_moe(const void *x, bool x_bf16, const int32_t *ids, const float *route_w,
                       int T, int topk, const int32_t *qw_gu, const float *sc_gu,
                       const int32_t *qw_dn, const float *sc_dn, int E, int H, int I,
                       int group, void *workspace, const float *shared_o, float *y,
                       cudaStream_t stream);

// ------------------------------------------------------------ MoE block
// Router: logits[T][E] = x W_r^T (fp32), then per token the topk experts by
// sigmoid(logit) + bias (bias may be nullptr), ties to the lower id, and
// weights scale * s_j / sum s (E <= 1024, topk <= 32).
cudaError_t launch_router(const void *x, bool x_bf16, int T, int H, const float *router_w,
                          const float *bias, int E, int topk, float scale, float *logits,
                          int32_t *ids, float *route_w, cudaStream_t stream);
// h[T][Is] = silu(gu[:, :Is]) * gu[:, Is:], bf16 or fp32.
cudaError_t launch_swiglu(const float *gu, int T, int Is, bool h_bf16, void *h,
                          cudaStream_t stream);

}  // namespace w4a16
