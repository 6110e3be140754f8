// Device and host helpers shared by the tcgen05 tensor-core kernels:
// shared-memory matrix descriptors, MMA issue and commit, TMEM loads, TMA
// tile loads, distributed shared memory within a cluster, and the driver's
// tensor-map encoder. sm_103a only.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

namespace w4a16 {
namespace tc {

// Shared-memory matrix descriptor for a K-major operand in the canonical
// 128-byte swizzled layout: 8-row x 128-byte atoms stacked at 1024-byte
// stride (SBO), start address in 16-byte units, descriptor version 1,
// swizzle mode 2 (128 B).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1) << 16;                 // LBO (unused for this layout)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;         // SBO
  d |= static_cast<uint64_t>(1) << 46;                 // version
  d |= static_cast<uint64_t>(2) << 61;                 // 128-byte swizzle
  return d;
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_mma(uint32_t dtmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(dtmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int c0, int c1,
                                            uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tmem_ld_32cols(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld_16cols(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Two fp32 -> packed bf16x2 (round to nearest even), lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// 8 packed nibbles (columns 0..7 of the word) * scale -> 8 bf16 in a uint4.
// (nibble - 8) is formed exactly as an fp32 (see nibble_pair), multiplied by
// the fp32 scale (one rounding, the format's own product), then rounded
// once more to bf16.
__device__ __forceinline__ uint4 dequant_word(uint32_t w, float s, const NibbleConsts &k) {
  const uint32_t w8 = w >> 8;
  const uint64_t p[4] = {nibble_pair<0>(w, w8, k), nibble_pair<1>(w, w8, k),
                         nibble_pair<2>(w, w8, k), nibble_pair<3>(w, w8, k)};
  // the odd nibble classes carry 16 (n - 8): scale them by s / 16 (exact,
  // a power-of-two scaling); one packed multiply per nibble pair
  const float so = s * nibble_prescale(1);
  uint64_t se2, so2;
  asm("mov.b64 %0, {%1, %1};" : "=l"(se2) : "f"(s));
  asm("mov.b64 %0, {%1, %1};" : "=l"(so2) : "f"(so));
  float lo[4], hi[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint64_t v;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(v) : "l"(p[c]), "l"((c & 1) ? so2 : se2));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo[c]), "=f"(hi[c]) : "l"(v));
  }
  uint4 o;
  o.x = pack_bf16x2(lo[0], lo[1]);
  o.y = pack_bf16x2(lo[2], lo[3]);
  o.z = pack_bf16x2(hi[0], hi[1]);
  o.w = pack_bf16x2(hi[2], hi[3]);
  return o;
}

// Store 32 consecutive TMEM columns of this warp's 32 lanes (one 32-bit
// value per lane and column); the caller waits with tmem_store_wait().
__device__ __forceinline__ void tmem_st_32cols(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st_16cols(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_store_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// MMA with the A operand in tensor memory (M = 128 lanes, K-major, two bf16
// per 32-bit column) and B in shared memory.
__device__ __forceinline__ void tc_mma_tmem_a(uint32_t dtmem, uint32_t atmem, uint64_t bdesc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(dtmem),
      "r"(atmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Load 16 bytes from the shared memory of cluster rank `rank` at the
// address of `p` in this CTA (p 16-byte aligned).
__device__ __forceinline__ float4 ld_cluster_f32x4(const float *p, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(a)
               : "memory");
  return v;
}

// Split-K reduction by the owner of a row slice. Every CTA of the cluster
// has parked its fp32 partial tile at red[row * LD + column] (BM columns) in
// its shared memory and passed a cluster barrier. This CTA owns rows
// lo .. lo + my_rows - 1: it reads 4 columns of a row from every rank
// (16-byte distributed shared-memory loads, all issued before the sums),
// adds them in rank order and stores y[m0 + m][n0 + row] for m0 + m < M and
// n0 + row < N. Consecutive threads take consecutive rows, so the y stores
// coalesce.
template <int BM, int LD, int MAXKS>
__device__ __forceinline__ void split_k_owner_reduce(const float *red, int lo, int my_rows, int ks,
                                                     int n0, int m0, int M, int N, void *y,
                                                     int ybf16) {
  for (int e = threadIdx.x; e < my_rows * (BM / 4); e += blockDim.x) {
    const int i = e % my_rows, c4 = e / my_rows;
    const int nl = lo + i;
    const float *src = red + nl * LD + 4 * c4;
    float4 part[MAXKS];
#pragma unroll
    for (int k = 0; k < MAXKS; ++k)
      if (k < ks) part[k] = ld_cluster_f32x4(src, static_cast<uint32_t>(k));
    float4 v = part[0];
#pragma unroll
    for (int k = 1; k < MAXKS; ++k)
      if (k < ks) {
        v.x += part[k].x; v.y += part[k].y; v.z += part[k].z; v.w += part[k].w;
      }
    if (n0 + nl >= N) continue;
    const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int m = 4 * c4 + t;
      if (m0 + m < M) store_y(y, static_cast<size_t>(m0 + m) * N + n0 + nl, vv[t], ybf16);
    }
  }
}

__device__ __forceinline__ bool aborted(const int *flag) {
  return *reinterpret_cast<const volatile int *>(flag) != 0;
}

// cuTensorMapEncodeTiled from the driver, looked up once.
inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

}  // namespace tc
}  // namespace w4a16
