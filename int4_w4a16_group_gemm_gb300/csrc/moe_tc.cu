// Grouped MoE expert GEMMs on the tcgen05 tensor cores (bf16 activations).
//
// "The Quiet Commit: How a Single Documentation Edit Marks the Completion of
// a Major Engineering Milestone", section "The Context: A Native DDTree
// Engine Takes Shape" (MoE experts with SwiGLU) and section "The INT4
// Milestone" (experts run through the W4A16 kernel).
//
// The same four steps as the CUDA-core layer (moe.cu), with the two expert
// GEMMs on the tensor cores:
//   gather:   the activation rows in expert-sorted order, xs[s] =
//             x[perm[s] / topk] (bf16), so that an expert's tokens are one
//             run of rows a TMA box can load;
//   gate/up:  per work unit (expert e, tile of up to 16 of its tokens, 64
//             rows of I) the MMA computes the tile's 64 gate rows and the
//             matching 64 up rows at once; h = silu(g) * u, stored per
//             sorted position as bf16;
//   down:     per unit (expert, token tile, 128 rows of H): o[pair] =
//             route_w[pair] * (h @ W_dn^T), stored per pair (fp32);
//   combine:  as in moe.cu.
// The product is computed transposed, D[row][token]: 128 weight rows are
// the MMA's M, the token tile (16) its N, so a unit's tensor work is small
// and its cost is the dequantisation, as in the small-M bf16 kernel
// (tc_split.cu), whose pipeline this kernel follows: the packed words and
// scales of each 256-column stage by TMA into a ring of 4 slots, 16
// dequantiser warps writing bf16 (nibble - 8) * scale into tensor memory,
// one warp issuing the MMAs warp-wide through an elected lane (A from TMEM,
// the token tile from shared memory), two accumulators so that the next
// unit's MMAs run while the current one is drained. CTAs are persistent
// over the units (expert-major, so the CTAs working at one time share an
// expert's token tile in L2).
// For gate/up, TMEM lane quadrant q holds gate rows 16q..16q+15 in its
// lanes 0..15 and the matching up rows in lanes 16..31, so each SwiGLU pair
// lies in one warp (a shuffle joins them). Every wait is bounded; a timeout
// is recorded in the status word and the CTA unwinds (TMEM is always freed).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "tc_core.cuh"

namespace w4a16 {

namespace {

using namespace tc;

constexpr int MX_BN = 16;           // tokens per unit (MMA N)
constexpr int MX_ROWS = 128;        // weight rows per unit (MMA M)
constexpr int MX_BK = 64;           // K columns per block
constexpr int MX_SK = 4;            // blocks per stage (one weight-ring slot)
constexpr int MX_NS = 3;            // stages of A (TMEM) and of the token tile (shared memory)
constexpr int MX_NW = 4;            // weight-ring slots
constexpr int MX_DQ_WARPS = 16;     // 4 blocks x 4 lane quadrants
constexpr int MX_WP_WARP = 2 + MX_DQ_WARPS;
constexpr int MX_THREADS = 96 + 32 * MX_DQ_WARPS;
constexpr int MX_W_BYTES = MX_ROWS * MX_SK * 32;      // 128 rows x 128 B
constexpr int MX_SC_BYTES = MX_ROWS * 8 * 4;          // 128 rows x up to 8 scales
constexpr int MX_WSLOT = MX_W_BYTES + MX_SC_BYTES;    // 20 KB
constexpr int MX_B_BYTES = MX_BN * MX_BK * 2;         // 2 KB per block
constexpr int MX_ACC = 2;                             // accumulators, MX_BN columns each
constexpr int MX_A_COL0 = 32;                         // first A block column
constexpr int MX_TMEM_COLS = 512;
constexpr int MX_RING_BYTES = MX_NS * MX_SK * MX_B_BYTES;  // 24 KB
constexpr int MX_WRING_BYTES = MX_NW * MX_WSLOT;           // 80 KB
constexpr int MX_SMEM = MX_RING_BYTES + MX_WRING_BYTES + 1024 + 256;
static_assert(MX_ACC * MX_BN <= MX_A_COL0, "accumulators below the A ring");
static_assert(MX_A_COL0 + MX_NS * MX_SK * 32 <= MX_TMEM_COLS, "TMEM budget");
static_assert(MX_WSLOT % 1024 == 0 && MX_B_BYTES % 1024 == 0 && MX_RING_BYTES % 1024 == 0,
              "128-byte swizzle atoms stay 1024-byte aligned");

// Instruction descriptor, kind::f16: D f32, A and B bf16, both K-major,
// N = 16, M = 128.
constexpr uint32_t MX_IDESC = (1u << 4) | (1u << 7) | (1u << 10) |
                              (static_cast<uint32_t>(MX_BN >> 3) << 17) |
                              (static_cast<uint32_t>(128 >> 4) << 24);

struct MxParams {
  const int32_t *offsets;  // [E + 1] expert offsets in sorted order
  const int32_t *items;    // work items (expert, token tile of MX_BN)
  const int32_t *n_items;
  const int32_t *perm;     // sorted position -> pair
  const float *route_w;    // [n] routing weights by pair
  void *out;               // gate/up: h bf16 [n][I] by sorted position; down: o fp32 [n][H] by pair
  int n_pairs, E, H, I;
  int K;       // reduced dimension: H (gate/up) or I (down)
  int tiles;   // row tiles per expert: I / 64 (gate/up) or H / 128 (down)
  int rows_e;  // weight rows per expert: 2 I (gate/up) or H (down)
  int gs;      // log2 of the group size
  int scb;     // floats per row in a stage's scale box: 8 (groups of 32) or 4
  int *status;
};

template <int MODE>
__global__ void __launch_bounds__(MX_THREADS, 1)
    moe_tc_kernel(const __grid_constant__ CUtensorMap tmap_b,
                  const __grid_constant__ CUtensorMap tmap_w,
                  const __grid_constant__ CUtensorMap tmap_s, const MxParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *wring = smem + MX_RING_BYTES;  // packed words (128-byte swizzle) + scales
  uint64_t *full = reinterpret_cast<uint64_t *>(wring + MX_WRING_BYTES);
  uint64_t *empty = full + MX_NS;
  uint64_t *wfull = empty + MX_NS;          // [MX_NW] slot landed
  uint64_t *wempty = wfull + MX_NW;         // [MX_NW] slot read
  uint64_t *acc_full = wempty + MX_NW;      // [MX_ACC] unit's MMAs complete
  uint64_t *acc_empty = acc_full + MX_ACC;  // [MX_ACC] unit drained
  uint64_t *drain = acc_empty + MX_ACC;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nstages = p.K / (MX_BK * MX_SK);  // the host admits K % 256 == 0 only
  const int units = *p.n_items * p.tiles;

  if (threadIdx.x == 0) {
    for (int s = 0; s < MX_NS; ++s) {
      mbar_init(&full[s], 1 + MX_DQ_WARPS);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < MX_NW; ++s) {
      mbar_init(&wfull[s], 1);
      mbar_init(&wempty[s], MX_DQ_WARPS);
    }
    for (int b = 0; b < MX_ACC; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);  // the 4 draining warps
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(MX_TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto fail = [&]() {
    record_status(p.status, W4A16_ERR_TIMEOUT);
    *reinterpret_cast<volatile int *>(abort_flag) = 1;
  };
  // unit u: row tile t of work item u / tiles (expert e, its sorted
  // positions [s0, s0 + mt)); false if the item is out of range
  auto unit_info = [&](int u, int &e, int &s0, int &mt, int &t) -> bool {
    const int it = u / p.tiles;
    t = u - it * p.tiles;
    e = p.items[2 * it];
    if (!W4A16_IN_BOUNDS(e >= 0 && e < p.E, p.status)) return false;
    s0 = p.offsets[e] + p.items[2 * it + 1] * MX_BN;
    mt = min(MX_BN, p.offsets[e + 1] - s0);
    return W4A16_IN_BOUNDS(s0 >= 0 && mt > 0 && s0 + mt <= p.n_pairs, p.status);
  };

  if (warp == 0) {
    // ------------------------------------------------ token tiles (TMA)
    if (lane == 0) {
      int st = 0;
      for (int u = blockIdx.x; u < units && !aborted(abort_flag); u += gridDim.x) {
        int e, s0, mt, t;
        if (!unit_info(u, e, s0, mt, t)) { fail(); break; }
        bool ok = true;
        for (int sg = 0; sg < nstages; ++sg, ++st) {
          const int s = st % MX_NS;
          const uint32_t ph = static_cast<uint32_t>(st / MX_NS) & 1u;
          if (!mbar_wait_backoff(&empty[s], ph ^ 1u, 32)) { fail(); ok = false; break; }
          mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(MX_SK * MX_B_BYTES));
          // rows s0 .. s0 + 15 (rows past the expert's tokens give columns
          // that are never stored; rows past n read as zero)
          for (int j = 0; j < MX_SK; ++j)
            tma_load_2d(smem + (s * MX_SK + j) * MX_B_BYTES, &tmap_b, (sg * MX_SK + j) * MX_BK, s0,
                        &full[s]);
        }
        if (!ok) break;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
    // the whole warp runs this loop (warp-uniform operands); one elected
    // lane issues
    int st = 0, ul = 0;
    bool issued_any = false;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++ul) {
      const int b = ul % MX_ACC;
      int got = 1;
      if (lane == 0)
        got = mbar_wait(&acc_empty[b], (static_cast<uint32_t>(ul / MX_ACC) & 1u) ^ 1u) &&
              !aborted(abort_flag);
      if (!__shfl_sync(0xFFFFFFFFu, got, 0)) {
        if (lane == 0) fail();
        break;
      }
      tc_fence_after();
      bool ok = true;
      for (int sg = 0; sg < nstages; ++sg, ++st) {
        const int s = st % MX_NS;
        const uint32_t ph = static_cast<uint32_t>(st / MX_NS) & 1u;
        got = 1;
        if (lane == 0) got = mbar_wait(&full[s], ph) && !aborted(abort_flag);
        if (!__shfl_sync(0xFFFFFFFFu, got, 0)) {
          if (lane == 0) fail();
          ok = false;
          break;
        }
        tc_fence_after();
        for (int j = 0; j < MX_SK; ++j) {
          const uint32_t a0 = tmem + MX_A_COL0 + (s * MX_SK + j) * 32;
          const uint64_t b0 = sw128_desc(smem_u32(smem + (s * MX_SK + j) * MX_B_BYTES));
#pragma unroll
          for (int k = 0; k < MX_BK / 16; ++k)  // +32 bytes per K step: +2 in the start field
            tc_mma_tmem_a_warp(tmem + b * MX_BN, a0 + k * 8, b0 + 2 * k, MX_IDESC,
                               (sg > 0 || j > 0 || k > 0) ? 1u : 0u);
        }
        tc_commit_warp(&empty[s]);
        issued_any = true;
      }
      if (!ok) break;
      tc_commit_warp(&acc_full[b]);
    }
    // every MMA this warp issued is complete before TMEM is released
    if (issued_any) {
      tc_commit_warp(drain);
      if (lane == 0) mbar_wait(drain, 0);
    }
    __syncwarp();
  } else if (warp == MX_WP_WARP) {
    // ------------------------------------------------- weight producer (TMA)
    // per stage two 64-row x 32-word boxes of packed words (gate/up: the 64
    // gate rows then the matching up rows; down: rows 0-63, 64-127) and the
    // two matching scale boxes, into a ring of MX_NW slots
    if (lane == 0) {
      int wit = 0;
      for (int u = blockIdx.x; u < units && !aborted(abort_flag); u += gridDim.x) {
        int e, s0, mt, t;
        if (!unit_info(u, e, s0, mt, t)) { fail(); break; }
        const int r0 = e * p.rows_e + (MODE == 0 ? 64 : 128) * t;
        const int r1 = MODE == 0 ? r0 + p.I : r0 + 64;
        bool ok = true;
        for (int sg = 0; sg < nstages; ++sg, ++wit) {
          const int ws = wit % MX_NW;
          const uint32_t wph = static_cast<uint32_t>(wit / MX_NW) & 1u;
          if (!mbar_wait_backoff(&wempty[ws], wph ^ 1u, 32)) { fail(); ok = false; break; }
          uint8_t *slot = wring + ws * MX_WSLOT;
          const int kb = sg * MX_SK;
          const int c0 = ((kb * MX_BK) >> p.gs) & ~3;  // first scale column, 16-byte aligned
          mbar_arrive_expect_tx(&wfull[ws], MX_W_BYTES + MX_ROWS * p.scb * 4);
          tma_load_2d(slot, &tmap_w, kb * 8, r0, &wfull[ws]);
          tma_load_2d(slot + MX_W_BYTES / 2, &tmap_w, kb * 8, r1, &wfull[ws]);
          tma_load_2d(slot + MX_W_BYTES, &tmap_s, c0, r0, &wfull[ws]);
          tma_load_2d(slot + MX_W_BYTES + 64 * p.scb * 4, &tmap_s, c0, r1, &wfull[ws]);
        }
        if (!ok) break;
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------- dequantisers
    const NibbleConsts nk_ = make_nibble_consts();
    const int j = (warp - 2) >> 2;  // block of the stage this warp fills
    const int q = warp & 3;         // TMEM lane quadrant of this warp
    // the slot row this thread's TMEM lane (MMA row q * 32 + lane) takes
    const int srow = MODE == 0 ? (lane < 16 ? 16 * q + lane : 64 + 16 * q + lane - 16)
                               : q * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const uint32_t wsw = static_cast<uint32_t>(srow & 7);
    const uint32_t woff0 = static_cast<uint32_t>(srow * 128) + (((2u * j) ^ wsw) << 4);
    const uint32_t woff1 = static_cast<uint32_t>(srow * 128) + (((2u * j + 1u) ^ wsw) << 4);
    (void)W4A16_IN_BOUNDS(woff1 + 16u <= static_cast<uint32_t>(MX_W_BYTES) &&
                              woff0 + 16u <= static_cast<uint32_t>(MX_W_BYTES),
                          p.status);
    int st = 0, wit = 0, ul = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++ul) {
      for (int sg = 0; sg < nstages; ++sg, ++st, ++wit) {
        const int s = st % MX_NS, ws = wit % MX_NW;
        const uint32_t ph = static_cast<uint32_t>(st / MX_NS) & 1u;
        const uint32_t wph = static_cast<uint32_t>(wit / MX_NW) & 1u;
        // the slot has landed, then the TMEM stage is free (one lane waits)
        int got = 1;
        if (lane == 0)
          got = mbar_wait_backoff(&wfull[ws], wph, 32) &&
                mbar_wait_backoff(&empty[s], ph ^ 1u, 32) && !aborted(abort_flag);
        got = __shfl_sync(0xFFFFFFFFu, got, 0);
        __syncwarp();  // orders lane 0's acquire before the other lanes' reads
        if (!got) { fail(); ok = false; break; }
        const uint8_t *wst = wring + ws * MX_WSLOT;
        const uint4 c0 = *reinterpret_cast<const uint4 *>(wst + woff0);
        const uint4 c1 = *reinterpret_cast<const uint4 *>(wst + woff1);
        // block sg * 4 + j, halves h: group ((sg * 4 + j) * 64 + 32 h) >> gs,
        // at its offset in the stage's aligned window of groups
        const float *ssl = reinterpret_cast<const float *>(wst + MX_W_BYTES) + srow * p.scb;
        const int cg = ((sg * MX_SK * MX_BK) >> p.gs) & ~3;
        float cs[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int off = ((((sg * MX_SK + j) * MX_BK) + 32 * h) >> p.gs) - cg;
          cs[h] = W4A16_IN_BOUNDS(off >= 0 && off < p.scb, p.status) ? ssl[off] : 0.f;
        }
        tc_fence_after();
        {
          uint32_t a[32];
          const uint32_t wv[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint4 d = dequant_word(wv[i], cs[i >> 2], nk_);
            a[4 * i] = d.x; a[4 * i + 1] = d.y; a[4 * i + 2] = d.z; a[4 * i + 3] = d.w;
          }
          tmem_st_32cols(lane_base + MX_A_COL0 + (s * MX_SK + j) * 32, a);
          tmem_store_wait();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&wempty[ws]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[s]);
      }
      if (!ok || j != 0) continue;
      // ------------------------------------------------ drain unit u (j == 0)
      const int b = ul % MX_ACC;
      int accd = 1;
      if (lane == 0)
        accd = mbar_wait(&acc_full[b], static_cast<uint32_t>(ul / MX_ACC) & 1u) &&
               !aborted(abort_flag);
      if (!__shfl_sync(0xFFFFFFFFu, accd, 0)) { fail(); ok = false; break; }
      tc_fence_after();
      uint32_t r[16];
      tmem_ld_16cols(lane_base + b * MX_BN, r);
      int e, s0, mt, t;
      const bool uok = unit_info(u, e, s0, mt, t);
      if (MODE == 0) {
        // lane i < 16: gate row 16q + i; lane i + 16: its up row
        const int col = 64 * t + 16 * q + lane;  // column of h (lanes < 16)
#pragma unroll
        for (int tok = 0; tok < MX_BN; ++tok) {
          const float v = __uint_as_float(r[tok]);
          const float up = __shfl_down_sync(0xFFFFFFFFu, v, 16);
          if (uok && lane < 16 && tok < mt &&
              W4A16_IN_BOUNDS(col < p.I && s0 + tok < p.n_pairs, p.status))
            static_cast<__nv_bfloat16 *>(p.out)[static_cast<size_t>(s0 + tok) * p.I + col] =
                __float2bfloat16_rn(silu_f(v) * up);
        }
      } else {
        const int row = 128 * t + q * 32 + lane;  // output column of o
#pragma unroll
        for (int tok = 0; tok < MX_BN; ++tok) {
          if (!uok || tok >= mt) continue;
          const int pair = p.perm[s0 + tok];
          if (W4A16_IN_BOUNDS(pair >= 0 && pair < p.n_pairs && row < p.H, p.status))
            static_cast<float *>(p.out)[static_cast<size_t>(pair) * p.H + row] =
                p.route_w[pair] * __uint_as_float(r[tok]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[b]);
    }
    __syncwarp();
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(MX_TMEM_COLS)
                 : "memory");
  }
}

// xs[s][:] = x[perm[s] / topk][:] (bf16 rows, 16-byte pieces).
__global__ void moe_gather_kernel(const uint16_t *__restrict__ x, const int32_t *__restrict__ perm,
                                  int n, int topk, int H, uint16_t *__restrict__ xs,
                                  int *status) {
  const int H8 = H >> 3;
  const long long total = static_cast<long long>(n) * H8;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int s = static_cast<int>(i / H8), c = static_cast<int>(i % H8);
    const int pr = perm[s];
    if (!W4A16_IN_BOUNDS(pr >= 0 && pr < n, status)) continue;
    reinterpret_cast<uint4 *>(xs + static_cast<size_t>(s) * H)[c] =
        reinterpret_cast<const uint4 *>(x + static_cast<size_t>(pr / topk) * H)[c];
  }
}

}  // namespace

bool moe_tc_supported(int n_pairs, int H, int I, int group) {
  const bool g = group == 32 || group == 64 || group == 128;
  return g && n_pairs >= MX_BN && H % 256 == 0 && I % 256 == 0 && (H / group) % 4 == 0 &&
         (I / group) % 4 == 0;
}

cudaError_t launch_moe_gather(const uint16_t *x, const int32_t *perm, int n, int topk, int H,
                              uint16_t *xs, cudaStream_t stream) {
  const DeviceInfo &di = device_info();
  const long long work = static_cast<long long>(n) * (H / 8);
  const int grid = static_cast<int>(std::min<long long>((work + 255) / 256, di.num_sms * 8ll));
  moe_gather_kernel<<<std::max(grid, 1), 256, 0, stream>>>(x, perm, n, topk, H, xs, di.status);
  return cudaGetLastError();
}

cudaError_t launch_moe_tc(int mode, const uint16_t *b, const int32_t *qw, const float *sc,
                          const int32_t *offsets, const int32_t *items, const int32_t *n_items,
                          const int32_t *perm, const float *route_w, int n_pairs, int E, int H,
                          int I, int group, int max_items, void *out, cudaStream_t stream) {
  const DeviceInfo &di = device_info();
  auto encode = encode_fn();
  if (encode == nullptr) return cudaErrorNotSupported;
  if (!moe_tc_supported(n_pairs, H, I, group)) return cudaErrorInvalidValue;
  MxParams p{};
  p.offsets = offsets;
  p.items = items;
  p.n_items = n_items;
  p.perm = perm;
  p.route_w = route_w;
  p.out = out;
  p.n_pairs = n_pairs;
  p.E = E;
  p.H = H;
  p.I = I;
  p.K = mode == 0 ? H : I;
  p.tiles = mode == 0 ? I / 64 : H / 128;
  p.rows_e = mode == 0 ? 2 * I : H;
  p.gs = group == 128 ? 7 : group == 64 ? 6 : 5;
  p.scb = group == 32 ? 8 : 4;
  p.status = di.status;
  const int K = p.K, G = K / group;
  const long long wrows = static_cast<long long>(E) * p.rows_e;
  const cuuint32_t estr[2] = {1, 1};
  // token tiles: rows of xs (gate/up) or h (down), bf16, 16 rows x 64
  // columns per box, 128-byte swizzle
  CUtensorMap tmap_b, tmap_w, tmap_s;
  const cuuint64_t bdims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(n_pairs)};
  const cuuint64_t bstr[1] = {static_cast<cuuint64_t>(K) * 2};
  const cuuint32_t bbox[2] = {MX_BK, MX_BN};
  CUresult r = encode(&tmap_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(b), bdims,
                      bstr, bbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  // packed words of every expert's rows [E * rows_e][K / 8], 64 rows x 32
  // words per box, 128-byte swizzle
  const cuuint64_t wdims[2] = {static_cast<cuuint64_t>(K / 8), static_cast<cuuint64_t>(wrows)};
  const cuuint64_t wstr[1] = {static_cast<cuuint64_t>(K / 8) * 4};
  const cuuint32_t wbox[2] = {MX_SK * 8, 64};
  r = encode(&tmap_w, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<int32_t *>(qw), wdims, wstr,
             wbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  // scales [E * rows_e][G], 64 rows x scb floats per box (an aligned window
  // of groups that holds the stage's)
  const cuuint64_t sdims[2] = {static_cast<cuuint64_t>(G), static_cast<cuuint64_t>(wrows)};
  const cuuint64_t sstr[1] = {static_cast<cuuint64_t>(G) * 4};
  const cuuint32_t sbox[2] = {static_cast<cuuint32_t>(p.scb), 64};
  r = encode(&tmap_s, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(sc), sdims, sstr,
             sbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;

  auto kern = mode == 0 ? moe_tc_kernel<0> : moe_tc_kernel<1>;
  static PerDeviceOnce attr_once[2];
  const cudaError_t attr_err = attr_once[mode ? 1 : 0].run(
      [&] { return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, MX_SMEM); });
  if (attr_err != cudaSuccess) return attr_err;
  const long long max_units = static_cast<long long>(max_items) * p.tiles;
  const int grid = static_cast<int>(std::max(1LL, std::min<long long>(max_units, di.num_sms)));
  kern<<<grid, MX_THREADS, MX_SMEM, stream>>>(tmap_b, tmap_w, tmap_s, p);
  return cudaGetLastError();
}

}  // namespace w4a16
