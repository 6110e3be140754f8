// w4a16_moe_gemm_noalloc: the grouped MoE layer with its scratch memory in a
// fixed device array that the library owns, for callers that cannot
// allocate device memory or hand the library a workspace.
//
// Who needs it: host code that may not allocate device memory once it is
// running - serving processes that reserve their whole device-memory budget
// at start-up, plugins whose host framework owns every allocation and
// offers no workspace, and code paths where a cudaMalloc would synchronise
// the device or take the allocator's lock at the wrong time. They still
// pass their own inputs and output; only the intermediate buffers come from
// here.
//
// The array is a file-scope __device__ variable, so every GPU that loads
// the library holds kNoAllocScratchBytes of it until the process exits. In
// host code its name is only a host-side stand-in, never a device address:
// the address is looked up once per device with cudaGetSymbolAddress, with
// that device current, on the first call made on that device.
#include <cuda_runtime.h>

#include <mutex>

#include "kernels.h"

namespace {

// 40 MiB: enough for 128 tokens x top-8 with hidden 7168 and expert width
// 2048 (about 37.4 MB of offsets, expert-sorted indices, SwiGLU outputs and
// per-slot expert outputs).
constexpr size_t kNoAllocScratchBytes = 40ull << 20;

__device__ __align__(256) unsigned char g_moe_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::once_flag g_scratch_once[kMaxDevices];
void *g_scratch_ptr[kMaxDevices];
cudaError_t g_scratch_err[kMaxDevices];

// Device address of the scratch array on the current device (set-up once
// per device, on the first call).
cudaError_t scratch_on_current_device(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::call_once(g_scratch_once[dev], [dev] {
    void *p = nullptr;
    g_scratch_err[dev] = cudaGetSymbolAddress(&p, g_moe_scratch);
    g_scratch_ptr[dev] = (g_scratch_err[dev] == cudaSuccess) ? p : nullptr;
  });
  *out = g_scratch_ptr[dev];
  return g_scratch_err[dev];
}

}  // namespace

extern "C" {

w4a16_status w4a16_moe_gemm_noalloc(const void *x, w4a16_act_dtype xdt,
                                    const int32_t *expert_ids, const float *route_w, int T,
                                    int topk, const int32_t *qw_gu, const float *sc_gu,
                                    const int32_t *qw_dn, const float *sc_dn, int E, int H, int I,
                                    int group, float *y, w4a16_stream_t stream) {
  if (T <= 0 || topk <= 0 || E <= 0 || H <= 0 || I <= 0) return W4A16_ERR_INVALID_ARG;
  // sizes whose intermediates do not fit the fixed array are rejected
  // before anything else happens
  if (w4a16_moe_workspace_size(T, topk, E, H, I) > kNoAllocScratchBytes)
    return W4A16_ERR_UNSUPPORTED;
  void *scratch = nullptr;
  if (scratch_on_current_device(&scratch) != cudaSuccess || scratch == nullptr)
    return W4A16_ERR_CUDA;
  // Nothing in the scratch needs to start at zero: every intermediate the
  // layer reads back is written earlier in the same call.
  return w4a16_moe_gemm(x, xdt, expert_ids, route_w, T, topk, qw_gu, sc_gu, qw_dn, sc_dn, E, H,
                        I, group, scratch, kNoAllocScratchBytes, y, stream);
}

}  // extern "C"
