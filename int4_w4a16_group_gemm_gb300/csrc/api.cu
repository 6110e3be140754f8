// C-ABI entry points of libw4a16.so: argument validation, kernel choice and
// the per-device status word. Declarations and contracts: include/w4a16.h.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "kernels.h"

// Per-device status word written by kernels (first error wins).
__device__ int g_w4a16_status;

namespace w4a16 {

namespace {
constexpr int kMaxDevices = 64;
DeviceInfo g_info[kMaxDevices];
std::once_flag g_once[kMaxDevices];
bool g_info_ok[kMaxDevices];

void init_device(int dev) {
  DeviceInfo &d = g_info[dev];
  d.device = dev;
  g_info_ok[dev] = false;
  if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return;
  if (cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
      cudaSuccess)
    return;
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_w4a16_status) != cudaSuccess) return;
  d.status = static_cast<int *>(p);
  g_info_ok[dev] = true;
}
}  // namespace

const DeviceInfo &device_info() {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= kMaxDevices) dev = 0;
  std::call_once(g_once[dev], init_device, dev);
  return g_info[dev];
}

namespace {
std::atomic<int> g_fault_next{0};
}

bool take_injected_fault() { return g_fault_next.exchange(0) != 0; }

static bool device_ready() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (dev < 0 || dev >= kMaxDevices) return false;
  device_info();
  return g_info_ok[dev];
}

}  // namespace w4a16

using namespace w4a16;

static inline bool aligned16(const void *p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

// Group sizes the kernels take: a lane's or a piece's columns (16 or 32)
// always lie inside one group.
static inline bool group_supported(int group) { return group == 32 || group == 64 || group == 128; }

static inline w4a16_status from_cuda(cudaError_t e) {
  return e == cudaSuccess ? W4A16_OK : W4A16_ERR_CUDA;
}

// M at or above which bf16 activations go to the tensor-core kernel, and
// from which (up to 64) fp32 activations go to the fp32-exact tensor-core
// kernel: the crossovers against the streaming kernel measured on the
// decode-sized weight (N = 4096, K = 7168).
static constexpr int kTcMinM = 4;
static constexpr int kTcF32MinM = 12;

enum class GemmKernel { Stream, Gemv, TensorBf16, TensorF32 };

// Kernel choice shared by the launch path and the launch-count query.
// Returns OK and sets *kind, or the rejection status.
static w4a16_status plan_gemm(int M, int N, int K, int group, w4a16_act_dtype xdt,
                              w4a16_algo algo, GemmKernel *kind) {
  if (M <= 0 || N <= 0 || K <= 0 || K % 32 != 0) return W4A16_ERR_INVALID_ARG;
  if (xdt != W4A16_ACT_F32 && xdt != W4A16_ACT_BF16) return W4A16_ERR_INVALID_ARG;
  if (algo != W4A16_ALGO_AUTO && algo != W4A16_ALGO_SIMT && algo != W4A16_ALGO_TC &&
      algo != W4A16_ALGO_STREAM && algo != W4A16_ALGO_GEMV)
    return W4A16_ERR_INVALID_ARG;
  if (!group_supported(group)) return W4A16_ERR_UNSUPPORTED;
  if (K % group != 0) return W4A16_ERR_INVALID_ARG;
  const bool bf16 = xdt == W4A16_ACT_BF16;
  const bool f32_tc_ok = !bf16 && tc_f32_supported(M, N, K) && K <= max_k_stream(1);
  const bool gemv_ok = gemv_supported(M, N, K, group);
  *kind = GemmKernel::Stream;
  if (algo == W4A16_ALGO_GEMV) {
    if (!gemv_ok) return W4A16_ERR_UNSUPPORTED;
    *kind = GemmKernel::Gemv;
  } else if (algo == W4A16_ALGO_TC) {
    if (bf16 && tc_gemm_supported(M, N, K))
      *kind = GemmKernel::TensorBf16;
    else if (f32_tc_ok)
      *kind = GemmKernel::TensorF32;
    else
      return W4A16_ERR_UNSUPPORTED;
  } else if (algo == W4A16_ALGO_AUTO) {
    if (bf16 && M >= kTcMinM && tc_gemm_supported(M, N, K))
      *kind = GemmKernel::TensorBf16;
    else if (f32_tc_ok && M >= kTcF32MinM)
      *kind = GemmKernel::TensorF32;
  }
  if (*kind == GemmKernel::Stream && K > max_k_stream(1)) return W4A16_ERR_UNSUPPORTED;
  return W4A16_OK;
}

extern "C" {

int w4a16_gemm_launches(int M, int N, int K, int group, w4a16_act_dtype xdt, w4a16_algo algo) {
  GemmKernel kind;
  const w4a16_status st = plan_gemm(M, N, K, group, xdt, algo, &kind);
  if (st != W4A16_OK) return -static_cast<int>(st);
  return kind == GemmKernel::Stream ? stream_gemm_passes(M, K) : 1;
}

w4a16_status w4a16_gemm_ex(const void *x, w4a16_act_dtype xdt, const int32_t *qw,
                           const float *sc, int M, int N, int K, int group, void *y,
                           w4a16_algo algo, unsigned int flags, w4a16_stream_t stream) {
  if (!x || !qw || !sc || !y) return W4A16_ERR_INVALID_ARG;
  if (flags & ~static_cast<unsigned int>(W4A16_FLAG_OVERLAP | W4A16_FLAG_OUT_BF16))
    return W4A16_ERR_INVALID_ARG;
  GemmKernel kind;
  const w4a16_status st = plan_gemm(M, N, K, group, xdt, algo, &kind);
  if (st != W4A16_OK) return st;
  if (!aligned16(x) || !aligned16(qw) || !aligned16(sc) || !aligned16(y))
    return W4A16_ERR_ALIGNMENT;
  if (!device_ready()) return W4A16_ERR_CUDA;
  const bool bf16 = xdt == W4A16_ACT_BF16;
  const bool overlap = (flags & W4A16_FLAG_OVERLAP) != 0;
  const bool ybf16 = (flags & W4A16_FLAG_OUT_BF16) != 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (kind == GemmKernel::TensorBf16)
    return from_cuda(launch_tc_gemm(static_cast<const uint16_t *>(x), qw, sc, M, N, K, group, y,
                                    ybf16, overlap, s));
  if (kind == GemmKernel::Gemv)
    return from_cuda(launch_gemv(x, bf16, qw, sc, N, K, group, y, ybf16, overlap, s));
  if (kind == GemmKernel::TensorF32)
    return from_cuda(launch_tc_f32(static_cast<const float *>(x), qw, sc, M, N, K, group, y,
                                   ybf16, overlap, s));
  return from_cuda(
      launch_stream_gemm(x, bf16, K, qw, sc, M, N, K, group, y, ybf16, N, overlap, s));
}

w4a16_status w4a16_gemm(const void *x, w4a16_act_dtype xdt, const int32_t *qw, const float *sc,
                        int M, int N, int K, int group, float *y, w4a16_stream_t stream) {
  return w4a16_gemm_ex(x, xdt, qw, sc, M, N, K, group, y, W4A16_ALGO_AUTO, 0u, stream);
}

w4a16_status w4a16_quantize(const float *w, int N, int K, int group, int32_t *qw, float *sc,
                            w4a16_stream_t stream) {
  if (!w || !qw || !sc) return W4A16_ERR_INVALID_ARG;
  if (N <= 0 || K <= 0 || K % 32 != 0) return W4A16_ERR_INVALID_ARG;
  if (!group_supported(group)) return W4A16_ERR_UNSUPPORTED;
  if (K % group != 0) return W4A16_ERR_INVALID_ARG;
  if (!aligned16(w) || !aligned16(qw)) return W4A16_ERR_ALIGNMENT;
  if (!device_ready()) return W4A16_ERR_CUDA;
  return from_cuda(
      launch_quantize(w, N, K, group, qw, sc, reinterpret_cast<cudaStream_t>(stream)));
}

w4a16_status w4a16_moe_sort(const int32_t *expert_ids, int n_pairs, int E, int32_t *offsets,
                            int32_t *perm, w4a16_stream_t stream) {
  if (!expert_ids || !offsets || !perm) return W4A16_ERR_INVALID_ARG;
  if (n_pairs < 0 || E <= 0) return W4A16_ERR_INVALID_ARG;
  if (E > 8192) return W4A16_ERR_UNSUPPORTED;
  if (!device_ready()) return W4A16_ERR_CUDA;
  return from_cuda(launch_moe_sort(expert_ids, n_pairs, E, offsets, perm,
                                   reinterpret_cast<cudaStream_t>(stream)));
}

size_t w4a16_moe_workspace_size(int T, int topk, int E, int H, int I) {
  if (T < 0 || topk <= 0 || E <= 0 || H <= 0 || I <= 0) return 0;
  return moe_workspace_bytes(T, topk, E, H, I);
}

w4a16_status w4a16_moe_workspace_layout(int T, int topk, int E, int H, int I, size_t *off_perm,
                                        size_t *off_h, size_t *off_o) {
  if (T <= 0 || topk <= 0 || E <= 0 || H <= 0 || I <= 0) return W4A16_ERR_INVALID_ARG;
  if (!off_perm || !off_h || !off_o) return W4A16_ERR_INVALID_ARG;
  moe_workspace_offsets(T, topk, E, H, I, off_perm, off_h, off_o);
  return W4A16_OK;
}

w4a16_status w4a16_moe_gemm(const void *x, w4a16_act_dtype xdt, const int32_t *expert_ids,
                            const float *route_w, int T, int topk, const int32_t *qw_gu,
                            const float *sc_gu, const int32_t *qw_dn, const float *sc_dn, int E,
                            int H, int I, int group, void *workspace, size_t ws_bytes, float *y,
                            w4a16_stream_t stream) {
  if (!x || !expert_ids || !route_w || !qw_gu || !sc_gu || !qw_dn || !sc_dn || !workspace || !y)
    return W4A16_ERR_INVALID_ARG;
  if (T <= 0 || topk <= 0 || E <= 0 || H <= 0 || I <= 0) return W4A16_ERR_INVALID_ARG;
  if (H % 32 != 0 || I % 32 != 0) return W4A16_ERR_INVALID_ARG;
  if (xdt != W4A16_ACT_F32 && xdt != W4A16_ACT_BF16) return W4A16_ERR_INVALID_ARG;
  if (!group_supported(group)) return W4A16_ERR_UNSUPPORTED;
  if (H % group != 0 || I % group != 0) return W4A16_ERR_INVALID_ARG;
  if (E > 8192 || H > max_k_stream(1) || I > max_k_stream(1)) return W4A16_ERR_UNSUPPORTED;
  if (ws_bytes < moe_workspace_bytes(T, topk, E, H, I)) return W4A16_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(qw_gu) || !aligned16(sc_gu) || !aligned16(qw_dn) ||
      !aligned16(sc_dn) || !aligned16(workspace) || !aligned16(y))
    return W4A16_ERR_ALIGNMENT;
  if (!device_ready()) return W4A16_ERR_CUDA;
  return from_cuda(launch_moe(x, xdt == W4A16_ACT_BF16, expert_ids, route_w, T, topk, qw_gu,
                              sc_gu, qw_dn, sc_dn, E, H, I, group, workspace, nullptr, y,
                              reinterpret_cast<cudaStream_t>(stream)));
}

static constexpr int kRouterMaxExperts = 1024;
static constexpr int kRouterMaxTopk = 32;

static w4a16_status check_router(const void *x, w4a16_act_dtype xdt, int T, int H,
                                 const float *router_w, int E, int topk, float route_scale) {
  if (!x || !router_w) return W4A16_ERR_INVALID_ARG;
  if (T <= 0 || H <= 0 || H % 32 != 0 || E <= 0 || topk <= 0 || topk > E)
    return W4A16_ERR_INVALID_ARG;
  if (xdt != W4A16_ACT_F32 && xdt != W4A16_ACT_BF16) return W4A16_ERR_INVALID_ARG;
  if (!(route_scale == route_scale) || route_scale == INFINITY || route_scale == -INFINITY)
    return W4A16_ERR_INVALID_ARG;
  if (E > kRouterMaxExperts || topk > kRouterMaxTopk) return W4A16_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(router_w)) return W4A16_ERR_ALIGNMENT;
  return W4A16_OK;
}

w4a16_status w4a16_moe_route(const void *x, w4a16_act_dtype xdt, int T, int H,
                             const float *router_w, const float *router_bias, int E, int topk,
                             float route_scale, float *logits, int32_t *expert_ids,
                             float *route_w, w4a16_stream_t stream) {
  const w4a16_status st = check_router(x, xdt, T, H, router_w, E, topk, route_scale);
  if (st != W4A16_OK) return st;
  if (!logits || !expert_ids || !route_w) return W4A16_ERR_INVALID_ARG;
  if (!device_ready()) return W4A16_ERR_CUDA;
  return from_cuda(launch_router(x, xdt == W4A16_ACT_BF16, T, H, router_w, router_bias, E, topk,
                                 route_scale, logits, expert_ids, route_w,
                                 reinterpret_cast<cudaStream_t>(stream)));
}

// Block workspace: the grouped layer's workspace, then the router logits
// [T][E], the shared expert's gate/up output [T][2 Is], its SwiGLU output
// [T][Is] and its down output [T][H] (fp32 each, 256-byte aligned).
struct BlockWs {
  size_t off_logits, off_gu, off_h, off_o, total;
};

static size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

static BlockWs block_ws(int T, int topk, int E, int H, int I, int Is) {
  BlockWs b{};
  const size_t t = static_cast<size_t>(T);
  b.off_logits = align256(moe_workspace_bytes(T, topk, E, H, I));
  b.off_gu = b.off_logits + align256(t * E * sizeof(float));
  b.off_h = b.off_gu + align256(t * 2 * Is * sizeof(float));
  b.off_o = b.off_h + align256(t * Is * sizeof(float));
  b.total = b.off_o + (Is > 0 ? align256(t * H * sizeof(float)) : 0);
  return b;
}

size_t w4a16_moe_block_workspace_size(int T, int topk, int E, int H, int I, int Is) {
  if (T < 0 || topk <= 0 || E <= 0 || H <= 0 || I <= 0 || Is < 0) return 0;
  return block_ws(T, topk, E, H, I, Is).total;
}

w4a16_status w4a16_moe_block(const void *x, w4a16_act_dtype xdt, int T, const float *router_w,
                             const float *router_bias, int E, int topk, float route_scale,
                             const int32_t *qw_gu, const float *sc_gu, const int32_t *qw_dn,
                             const float *sc_dn, int H, int I, const int32_t *qw_sgu,
                             const float *sc_sgu, const int32_t *qw_sdn, const float *sc_sdn,
                             int Is, int group, void *workspace, size_t ws_bytes,
                             int32_t *expert_ids, float *route_w, float *y,
                             w4a16_stream_t stream) {
  w4a16_status st = check_router(x, xdt, T, H, router_w, E, topk, route_scale);
  if (st != W4A16_OK) return st;
  if (!qw_gu || !sc_gu || !qw_dn || !sc_dn || !workspace || !expert_ids || !route_w || !y)
    return W4A16_ERR_INVALID_ARG;
  if (I <= 0 || I % 32 != 0 || Is < 0 || Is % 32 != 0) return W4A16_ERR_INVALID_ARG;
  if (Is > 0 && (!qw_sgu || !sc_sgu || !qw_sdn || !sc_sdn)) return W4A16_ERR_INVALID_ARG;
  if (!group_supported(group)) return W4A16_ERR_UNSUPPORTED;
  if (H % group != 0 || I % group != 0 || Is % group != 0) return W4A16_ERR_INVALID_ARG;
  if (H > max_k_stream(1) || I > max_k_stream(1) || Is > max_k_stream(1))
    return W4A16_ERR_UNSUPPORTED;
  const BlockWs L = block_ws(T, topk, E, H, I, Is);
  if (ws_bytes < L.total) return W4A16_ERR_INVALID_ARG;
  if (!aligned16(qw_gu) || !aligned16(sc_gu) || !aligned16(qw_dn) || !aligned16(sc_dn) ||
      !aligned16(workspace) || !aligned16(y))
    return W4A16_ERR_ALIGNMENT;
  if (Is > 0 && (!aligned16(qw_sgu) || !aligned16(sc_sgu) || !aligned16(qw_sdn) ||
                 !aligned16(sc_sdn)))
    return W4A16_ERR_ALIGNMENT;
  if (!device_ready()) return W4A16_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  const bool bf16 = xdt == W4A16_ACT_BF16;

  // 1. router: logits, top-k ids and weights (into the caller's buffers)
  st = from_cuda(launch_router(x, bf16, T, H, router_w, router_bias, E, topk, route_scale,
                               reinterpret_cast<float *>(ws + L.off_logits), expert_ids, route_w,
                               s));
  if (st != W4A16_OK) return st;
  // 2. shared expert: gate/up GEMM, SwiGLU, down GEMM (each GEMM on the
  //    kernel its token count selects)
  float *shared_o = nullptr;
  if (Is > 0) {
    float *gu = reinterpret_cast<float *>(ws + L.off_gu);
    void *h = ws + L.off_h;
    shared_o = reinterpret_cast<float *>(ws + L.off_o);
    st = w4a16_gemm_ex(x, xdt, qw_sgu, sc_sgu, T, 2 * Is, H, group, gu, W4A16_ALGO_AUTO, 0u,
                       stream);
    if (st != W4A16_OK) return st;
    st = from_cuda(launch_swiglu(gu, T, Is, bf16, h, s));
    if (st != W4A16_OK) return st;
    st = w4a16_gemm_ex(h, xdt, qw_sdn, sc_sdn, T, H, Is, group, shared_o, W4A16_ALGO_AUTO, 0u,
                       stream);
    if (st != W4A16_OK) return st;
  }
  // 3. routed experts: sort, gate/up + SwiGLU, down x weight, combine (+ shared)
  return from_cuda(launch_moe(x, bf16, expert_ids, route_w, T, topk, qw_gu, sc_gu, qw_dn, sc_dn,
                              E, H, I, group, ws, shared_o, y, s));
}

void w4a16_debug_fault_next_launch(int enable) { w4a16::g_fault_next.store(enable ? 1 : 0); }

const char *w4a16_status_string(w4a16_status s) {
  switch (s) {
    case W4A16_OK: return "W4A16_OK";
    case W4A16_ERR_INVALID_ARG: return "W4A16_ERR_INVALID_ARG";
    case W4A16_ERR_UNSUPPORTED: return "W4A16_ERR_UNSUPPORTED";
    case W4A16_ERR_ALIGNMENT: return "W4A16_ERR_ALIGNMENT";
    case W4A16_ERR_CUDA: return "W4A16_ERR_CUDA";
    case W4A16_ERR_TIMEOUT: return "W4A16_ERR_TIMEOUT";
    case W4A16_ERR_BOUNDS: return "W4A16_ERR_BOUNDS";
  }
  return "W4A16_ERR_UNKNOWN";
}

w4a16_status w4a16_last_device_status(w4a16_stream_t stream) {
  if (!device_ready()) return W4A16_ERR_CUDA;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return W4A16_ERR_CUDA;
  int v = 0;
  const DeviceInfo &d = device_info();
  if (cudaMemcpy(&v, d.status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return W4A16_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpy(d.status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
    return W4A16_ERR_CUDA;
  return static_cast<w4a16_status>(v);
}

}  // extern "C"
