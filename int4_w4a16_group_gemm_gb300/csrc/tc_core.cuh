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

// L2 eviction policy (createpolicy) for cache-hinted loads: evict_last
// keeps a line in L2 ahead of normally cached lines.
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// tma_load_2d with an L2 cache policy.
__device__ __forceinline__ void tma_load_2d_hint(void *dst, const CUtensorMap *map, int c0, int c1,
                                                 uint64_t *bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(policy)
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

// Warp-wide forms of MMA issue and commit: every lane of a converged warp
// executes them with the same operands and one elected lane issues. Run
// from a single-lane branch, each MMA first moves its operands into uniform
// registers, which makes issue slower than the tensor core at N = 64 and
// several times slower again while other warps compete for issue slots; a
// warp-uniform issuing loop keeps the operands uniform.
__device__ __forceinline__ void tc_mma_tmem_a_warp(uint32_t dtmem, uint32_t atmem, uint64_t bdesc,
                                                   uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(dtmem),
      "r"(atmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tc_mma_warp(uint32_t dtmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(dtmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tc_commit_warp(uint64_t *bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          smem_u32(bar))
      : "memory");
}

// ------------------------------------------------ split-K reduction by push
// A tile of ROWS weight rows x BM tokens is split over K across the ks CTAs
// (ranks) of a cluster; rank r owns the row slice [r R, (r + 1) R), R = ROWS / ks.
// Every rank parks its fp32 partial tile at red[row * LD + column] in its
// own shared memory and sends each other rank that rank's slice with one
// bulk shared -> shared copy (the copy engine moves it; completion is
// counted in bytes on the owner's mbarrier). The owner adds the ks partials
// of its slice in rank order, so the result does not depend on timing.
// Received slices go to a dedicated buffer (slot k < r for sender k < r,
// k - 1 otherwise), never to memory the owner may still be using.
//
// Protocol (all waits bounded):
//   set-up   one thread: mbar_init(bar, 1); push_expect(bar, ks); the
//            barrier inits are fenced (fence_mbar_init) and then every
//            thread does cluster_arrive() (phase A);
//   end      every thread: cluster_wait() (phase A: every rank's barrier
//            is initialised), then one thread push_send(); every thread
//            waits for `bar`, cluster_arrive() (phase B: this rank has
//            received), push_owner_sum(), cluster_wait() (phase B: every
//            copy this CTA sent has landed, so its shared memory may go).
// Relaxed arrive: neither phase publishes ordinary stores (the barrier
// inits are published by fence_mbar_init, the slices by the copy engine's
// byte count), and a release here waits for every outstanding store of the
// thread.
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of this CTA's shared-memory word `saddr` in the CTA of cluster
// rank `rank`.
__device__ __forceinline__ uint32_t cluster_map(uint32_t saddr, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(saddr), "r"(rank));
  return a;
}

// ks is a power of two (1 .. MAXKS) that divides ROWS: slices are equal,
// ROWS >> log2(ks) rows each, and no division is needed.
__device__ __forceinline__ int log2_pow2(int v) { return __ffs(v) - 1; }

// Bytes of the receive buffer for clusters of up to MAXKS ranks.
template <int ROWS, int LD, int MAXKS>
constexpr int push_recv_bytes() {
  static_assert(ROWS % MAXKS == 0, "equal slices");
  return MAXKS > 1 ? (MAXKS - 1) * (ROWS / MAXKS) * LD * 4 : 16;
}

// Arm the owner's barrier for the ks - 1 incoming slices of its rows
// (called once, right after mbar_init(bar, 1)).
template <int ROWS, int LD>
__device__ __forceinline__ void push_expect(uint64_t *bar, int ks) {
  const int rows = ROWS >> log2_pow2(ks);
  mbar_arrive_expect_tx(bar, static_cast<uint32_t>((ks - 1) * rows * LD * 4));
}

// Send every other rank its slice of this rank's parked tile. The tile's
// writers have fenced their stores to the async proxy and passed a CTA
// barrier. Slices start on 16-byte boundaries (LD * 4 a multiple of 16).
template <int ROWS, int LD>
__device__ __forceinline__ void push_send(const float *red, float *recv, uint64_t *bar, int rank,
                                          int ks) {
  const int rows = ROWS >> log2_pow2(ks);
  for (int r = 0; r < ks; ++r) {
    if (r == rank) continue;
    const int k = rank < r ? rank : rank - 1;  // slot of this rank at the owner
    const uint32_t dst = cluster_map(smem_u32(recv + k * rows * LD), static_cast<uint32_t>(r));
    const uint32_t rbar = cluster_map(smem_u32(bar), static_cast<uint32_t>(r));
    asm volatile(
        "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, "
        "[%3];" ::"r"(dst),
        "r"(smem_u32(red + r * rows * LD)), "r"(static_cast<uint32_t>(rows * LD * 4)), "r"(rbar)
        : "memory");
  }
}

// The owner's sum: rows [lo, lo + rows) of the tile, lo = rank * rows, the
// ks partials (own parked tile for k == rank, receive slot otherwise) added
// in rank order; y[m0 + m][n0 + row] written for m0 + m < M and
// n0 + row < N. Consecutive threads take consecutive rows, so the y stores
// coalesce.
template <int ROWS, int BM, int LD, int MAXKS>
__device__ __forceinline__ void push_owner_sum(const float *red, const float *recv, int rank, int ks,
                                               int n0, int m0, int M, int N, void *y, int ybf16,
                                               int *status) {
  const int lrows = log2_pow2(ROWS) - log2_pow2(ks), rows = 1 << lrows;
  const int lo = rank * rows;
  for (int e = threadIdx.x; e < rows * (BM / 4); e += blockDim.x) {
    const int i = e & (rows - 1), c4 = e >> lrows;
    float4 part[MAXKS];
#pragma unroll
    for (int k = 0; k < MAXKS; ++k)
      if (k < ks) {
        const float *src = k == rank ? red + (lo + i) * LD
                                     : recv + ((k < rank ? k : k - 1) * rows + i) * LD;
        part[k] = *reinterpret_cast<const float4 *>(src + 4 * c4);
      }
    float4 v = part[0];
#pragma unroll
    for (int k = 1; k < MAXKS; ++k)
      if (k < ks) {
        v.x += part[k].x; v.y += part[k].y; v.z += part[k].z; v.w += part[k].w;
      }
    if (n0 + lo + i >= N) continue;
    const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int m = 4 * c4 + t;
      if (m0 + m < M && W4A16_IN_BOUNDS(m0 + m >= 0 && n0 + lo + i >= 0, status))
        store_y(y, static_cast<size_t>(m0 + m) * N + n0 + lo + i, vv[t], ybf16);
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
