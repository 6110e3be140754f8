// Small-M W4A16 GEMM on the tcgen05 tensor cores (bf16 activations), with
// the dequantised weights kept in tensor memory and K split over a cluster.
//
//   y[m][n] = sum_k x[m][k] * W_hat[n][k],  W_hat = (nibble - 8) * scale
//
// As in the large-M kernel the product is computed transposed, D[n][m]: the
// 128 weight rows of a tile are the MMA's M, 64 tokens its N. At this size
// the dequantised A tile is the bandwidth problem: written to shared memory
// by the CUDA cores and read back by every MMA, it costs 4 bytes of
// shared-memory traffic per weight, which is what bounds a shared-memory-A
// kernel here. So the dequantisers store A straight into tensor memory
// (tcgen05.st) and the MMAs read it from there (the A-in-TMEM form of
// tcgen05.mma); shared memory only carries the activations (TMA).
//
// Tile: 128 weight rows x 64 tokens, K split over a cluster of ks CTAs
// (grid y = rank) at whole stages. Pipeline stage = 4 blocks of 64 K
// columns, 3 stages:
//   warp 0       TMA: one 64 x 64 bf16 activation box (128-byte swizzle)
//                per block into the stage's B slot;
//   warp 1       TMEM owner and MMA issuer: per stage, 4 x 4 MMAs
//                (M=128, N=64, K=16) with A from TMEM, one commit, issued
//                warp-wide by an elected lane;
//   warps 2-17   dequantisers: warp w handles block (w - 2) / 4 of every
//                stage for TMEM lane quadrant w % 4; thread = weight row,
//                8 packed words (64 columns) per block and the row's two
//                group scales, read from the weight ring, dequantised to
//                bf16 pairs and stored as 32 TMEM columns;
//   warp 18      weight producer: one TMA box of the stage's packed words
//                (128 rows x 128 bytes, 128-byte swizzle) and one of its
//                scales (128 rows x 8 or 4 floats) into a ring of 4, so the
//                weight stream runs ahead with few, large requests. (When
//                a scale row is not a whole number of 16-byte units the
//                dequantisers load their scales themselves, two stages
//                ahead.)
// TMEM: columns 0-63 the fp32 accumulator, 64 + 32 * (stage * 4 + block)
// the A blocks (448 of 512 columns).
// Epilogue: each rank parks its fp32 partial tile in shared memory and
// pushes every other rank's row slice to it with one bulk shared -> shared
// copy; the owner of a slice adds the partials in rank order, so the result
// is deterministic and needs no workspace (split-K helpers, tc_core.cuh).
// Every wait is bounded; a timeout is recorded in the status word and the
// CTA unwinds (TMEM is always freed).
//
// Format: "The Quiet Commit: How a Single Documentation Edit Marks the
// Completion of a Major Engineering Milestone", section "The INT4 Milestone".
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "tc_core.cuh"

namespace w4a16 {

namespace {

using namespace tc;

constexpr int SP_BM = 64;          // tokens per tile (MMA N)
constexpr int SP_ROWS = 128;       // weight rows per tile (MMA M)
constexpr int SP_BK = 64;          // K columns per block
constexpr int SP_SK = 4;           // blocks per stage
constexpr int SP_NS = 3;           // stages
constexpr int SP_DQ_WARPS = 16;    // 4 blocks x 4 lane quadrants
constexpr int SP_WP_WARP = 2 + SP_DQ_WARPS;  // the weight producer (TMA)
constexpr int SP_THREADS = 96 + 32 * SP_DQ_WARPS;
constexpr int SP_NW = 4;           // stages of packed weights in shared memory
constexpr int SP_W_BYTES = SP_ROWS * SP_SK * 32;  // 128 rows x 128 B per stage
// scales of a stage (scales by TMA): 128 rows x SCB floats, SCB = 8 for
// groups of 32 (the stage's 8 groups), 4 otherwise (an aligned window that
// holds the stage's 4, 2 groups)
constexpr int SP_SC_BYTES = SP_ROWS * 8 * 4;
constexpr int SP_WSLOT = SP_W_BYTES + SP_SC_BYTES;  // one weight-ring slot
constexpr int SP_B_BYTES = SP_BM * SP_BK * 2;               // 8 KB per block
constexpr int SP_ACC_COLS = SP_BM;                          // fp32 accumulator
constexpr int SP_A_COL0 = SP_ACC_COLS;                      // first A block column
constexpr int SP_TMEM_COLS = 512;
constexpr int SP_RING_BYTES = SP_NS * SP_SK * SP_B_BYTES;   // 96 KB
constexpr int SP_WRING_BYTES = SP_NW * SP_WSLOT;           // 80 KB
constexpr int SP_RED_LD = SP_BM + 4;  // row stride of the parked partial tile (floats)
constexpr int SP_MAX_KS = 8;          // largest cluster (K split)
constexpr int SP_RECV_BYTES = push_recv_bytes<SP_ROWS, SP_RED_LD, SP_MAX_KS>();
constexpr int SP_SMEM = SP_RING_BYTES + SP_WRING_BYTES + SP_RECV_BYTES + 1024 + 256;
static_assert(SP_A_COL0 + SP_NS * SP_SK * 32 <= SP_TMEM_COLS, "TMEM budget");
static_assert(SP_ROWS * (SP_BM + 4) * 4 <= SP_RING_BYTES, "parked partial tile");
static_assert(SP_WSLOT % 1024 == 0, "weight slots keep the 128-byte swizzle atoms aligned");

// Instruction descriptor, kind::f16: D f32, A and B bf16, both K-major,
// N = 64, M = 128.
constexpr uint32_t SP_IDESC = (1u << 4) | (1u << 7) | (1u << 10) |
                              (static_cast<uint32_t>(SP_BM >> 3) << 17) |
                              (static_cast<uint32_t>(128 >> 4) << 24);

struct SpParams {
  const int32_t *qw;
  const float *sc;
  void *y;  // fp32, or bf16 when ybf16
  int ybf16;
  int M, N, K;
  int gs;   // log2 of the group size
  int lks;  // log2 of the K split (cluster size)
  int scb;  // floats per row in a stage's scale box (scales by TMA)
  int *status;
};

// SCT: the scales come by TMA with the packed words (a box of 128 rows x
// scb floats per stage); otherwise each dequantiser thread loads its row's
// scales from global memory two stages ahead (the scale rows must then
// have a 16-byte multiple stride for the tensor map, K / group % 4 == 0).
// Grid: x = weight-row tile, y = K rank (the cluster), z = token tile.
template <bool SCT>
__global__ void __launch_bounds__(SP_THREADS, 1)
    tc_split_kernel(const __grid_constant__ CUtensorMap tmap_x,
                    const __grid_constant__ CUtensorMap tmap_w,
                    const __grid_constant__ CUtensorMap tmap_s, const SpParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *wring = smem + SP_RING_BYTES;  // packed weights, 128-byte swizzle
  float *recv = reinterpret_cast<float *>(wring + SP_WRING_BYTES);  // split-K slices received
  uint64_t *full = reinterpret_cast<uint64_t *>(wring + SP_WRING_BYTES + SP_RECV_BYTES);
  uint64_t *empty = full + SP_NS;
  uint64_t *wfull = empty + SP_NS;     // [SP_NW] packed weights (and scales) landed
  uint64_t *wempty = wfull + SP_NW;    // [SP_NW] packed weights read
  uint64_t *acc_full = wempty + SP_NW;
  uint64_t *drain = acc_full + 1;
  uint64_t *red_bar = drain + 1;       // split-K slices of this rank's rows landed
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(red_bar + 1);
  int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = p.K;
  const int nk = (K + SP_BK - 1) / SP_BK;
  // K is split at whole stages: rank r takes stages [nst r / ks, nst (r+1) / ks)
  // (the launcher keeps ks <= nst, so every rank has at least one)
  const int nst = (nk + SP_SK - 1) / SP_SK;
  const int rank = static_cast<int>(blockIdx.y);
  const int ks = 1 << p.lks;
  const int kb0 = ((nst * rank) >> p.lks) * SP_SK;
  const int kb1 = min(nk, ((nst * (rank + 1)) >> p.lks) * SP_SK);
  const int n0 = static_cast<int>(blockIdx.x) * SP_ROWS;
  const int m0 = static_cast<int>(blockIdx.z) * SP_BM;

  if (threadIdx.x == 0) {
    for (int s = 0; s < SP_NS; ++s) {
      mbar_init(&full[s], 1 + SP_DQ_WARPS);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < SP_NW; ++s) {
      mbar_init(&wfull[s], 1);
      mbar_init(&wempty[s], SP_DQ_WARPS);
    }
    mbar_init(acc_full, 1);
    mbar_init(drain, 1);
    mbar_init(red_bar, 1);
    if (ks > 1) push_expect<SP_ROWS, SP_RED_LD>(red_bar, ks);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(SP_TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_arrive();  // phase A: this rank's barriers are initialised
  const uint32_t tmem = *tmem_slot;
  // Programmatic launch: the weights are read before griddep_wait (never
  // written by the previous kernel, by the overlap contract), x and y after.
  griddep_launch_dependents();

  auto fail = [&]() {
    record_status(p.status, W4A16_ERR_TIMEOUT);
    *reinterpret_cast<volatile int *>(abort_flag) = 1;
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA
    if (lane == 0) {
      griddep_wait();
      int it = 0;
      for (int kb = kb0; kb < kb1 && !aborted(abort_flag); kb += SP_SK, ++it) {
        const int s = it % SP_NS;
        const uint32_t ph = static_cast<uint32_t>(it / SP_NS) & 1u;
        const int nsub = min(SP_SK, kb1 - kb);
        if (!mbar_wait_backoff(&empty[s], ph ^ 1u, 32)) { fail(); break; }
        if (aborted(abort_flag)) break;
        mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(nsub * SP_B_BYTES));
        for (int j = 0; j < nsub; ++j)
          tma_load_2d(smem + (s * SP_SK + j) * SP_B_BYTES, &tmap_x, (kb + j) * SP_BK, m0,
                      &full[s]);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
    // the whole warp runs this loop (warp-uniform operands); one elected
    // lane issues (tc_mma_tmem_a_warp)
    int it = 0;
    bool issued_any = false, ok = true;
    for (int kb = kb0; kb < kb1; kb += SP_SK, ++it) {
      const int s = it % SP_NS;
      const uint32_t ph = static_cast<uint32_t>(it / SP_NS) & 1u;
      const int nsub = min(SP_SK, kb1 - kb);
      int got = 1;
      if (lane == 0) got = mbar_wait(&full[s], ph) && !aborted(abort_flag);
      if (!__shfl_sync(0xFFFFFFFFu, got, 0)) {
        if (lane == 0) fail();
        ok = false;
        break;
      }
      tc_fence_after();
      for (int j = 0; j < nsub; ++j) {
        const uint32_t a0 = tmem + SP_A_COL0 + (s * SP_SK + j) * 32;
        const uint64_t b0 = sw128_desc(smem_u32(smem + (s * SP_SK + j) * SP_B_BYTES));
#pragma unroll
        for (int k = 0; k < SP_BK / 16; ++k)  // +32 bytes per K step: +2 in the start field
          tc_mma_tmem_a_warp(tmem, a0 + k * 8, b0 + 2 * k, SP_IDESC,
                             (kb + j > kb0 || k > 0) ? 1u : 0u);
      }
      tc_commit_warp(&empty[s]);
      issued_any = true;
    }
    if (ok) tc_commit_warp(acc_full);
    // all MMAs this warp issued are complete before TMEM is released
    if (issued_any) {
      tc_commit_warp(drain);
      if (lane == 0) mbar_wait(drain, 0);
    }
    __syncwarp();
  } else if (warp == SP_WP_WARP) {
    // ------------------------------------------------- weight producer (TMA)
    // one 128-row x 32-word box per stage (the 4 blocks' packed words;
    // words past K read as zero), 128-byte swizzle, and with SCT the
    // stage's scale box; runs SP_NW stages ahead
    if (lane == 0) {
      int it = 0;
      for (int kb = kb0; kb < kb1 && !aborted(abort_flag); kb += SP_SK, ++it) {
        const int ws = it % SP_NW;
        const uint32_t ph = static_cast<uint32_t>(it / SP_NW) & 1u;
        if (!mbar_wait_backoff(&wempty[ws], ph ^ 1u, 32)) { fail(); break; }
        if (aborted(abort_flag)) break;
        uint8_t *slot = wring + ws * SP_WSLOT;
        if constexpr (SCT) {
          // the stage's scales: groups from ((kb * 64) >> gs) aligned down to 4
          mbar_arrive_expect_tx(&wfull[ws], SP_W_BYTES + SP_ROWS * p.scb * 4);
          tma_load_2d(slot + SP_W_BYTES, &tmap_s, ((kb * SP_BK) >> p.gs) & ~3, n0, &wfull[ws]);
        } else {
          mbar_arrive_expect_tx(&wfull[ws], SP_W_BYTES);
        }
        tma_load_2d(slot, &tmap_w, kb * 8, n0, &wfull[ws]);
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------- dequantisers
    const NibbleConsts nk_ = make_nibble_consts();
    const int dw = warp - 2;
    const int j = dw >> 2;                 // block of the stage this warp fills
    const int q = warp & 3;                // TMEM lane quadrant of this warp
    const int row = q * 32 + lane;         // weight row within the tile = TMEM lane
    const int n = n0 + row;
    const bool nvalid = n < p.N;
    const int Kw = K >> 3;
    const int G = K >> p.gs;
    const float *srow = p.sc + static_cast<size_t>(nvalid ? n : 0) * G;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
    // this row's two scales of block kb (0 past K or N), from global memory
    auto fetch_sc = [&](int kb, float (&sc)[2]) {
      sc[0] = sc[1] = 0.f;
      if (SCT || !nvalid || kb >= kb1) return;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int w0 = kb * 8 + 4 * h;
        if (w0 < Kw && W4A16_IN_BOUNDS(((w0 * 8) >> p.gs) < G, p.status))
          sc[h] = __ldg(srow + ((w0 * 8) >> p.gs));  // 32 columns, one group
      }
    };
    // this row's 16-byte chunks 2j and 2j+1 in a weight stage (row r at
    // r * 128 bytes, chunk c at (c ^ (r & 7)) * 16)
    const uint32_t wsw = static_cast<uint32_t>(row & 7);
    const uint32_t woff0 = static_cast<uint32_t>(row * 128) + (((2u * j) ^ wsw) << 4);
    const uint32_t woff1 = static_cast<uint32_t>(row * 128) + (((2u * j + 1u) ^ wsw) << 4);
    (void)W4A16_IN_BOUNDS(woff0 + 16u <= static_cast<uint32_t>(SP_W_BYTES) &&
                              woff1 + 16u <= static_cast<uint32_t>(SP_W_BYTES),
                          p.status);
    float rsc[2][2];
    fetch_sc(kb0 + j, rsc[0]);
    fetch_sc(kb0 + SP_SK + j, rsc[1]);
    int it = 0;
    bool ok = true;
    for (int kbase = kb0; kbase < kb1 && ok; kbase += 2 * SP_SK) {
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int kbs = kbase + u * SP_SK;  // first block of the stage
        if (kbs >= kb1) break;
        const int s = it % SP_NS, ws = it % SP_NW;
        const uint32_t ph = static_cast<uint32_t>(it / SP_NS) & 1u;
        const uint32_t wph = static_cast<uint32_t>(it / SP_NW) & 1u;
        ++it;
        float cs[2] = {rsc[u][0], rsc[u][1]};
        fetch_sc(kbs + 2 * SP_SK + j, rsc[u]);
        // the packed words have landed, then the TMEM slot is free
        // (one lane waits, sleeping between polls: these warps run ahead of
        // the MMA warp, which shares their schedulers)
        int got = 1;
        if (lane == 0)
          got = mbar_wait_backoff(&wfull[ws], wph, 32) &&
                mbar_wait_backoff(&empty[s], ph ^ 1u, 32) && !aborted(abort_flag);
        got = __shfl_sync(0xFFFFFFFFu, got, 0);
        __syncwarp();  // orders lane 0's acquire before the other lanes' reads
        if (!got) { fail(); ok = false; break; }
        const uint8_t *wst = wring + ws * SP_WSLOT;
        const uint4 c0 = *reinterpret_cast<const uint4 *>(wst + woff0);
        const uint4 c1 = *reinterpret_cast<const uint4 *>(wst + woff1);
        if constexpr (SCT) {
          // block kbs + j, halves h: group ((kbs + j) * 64 + 32 h) >> gs,
          // at its offset in the stage's aligned window of groups
          const float *srow_s = reinterpret_cast<const float *>(wst + SP_W_BYTES) + row * p.scb;
          const int c0g = ((kbs * SP_BK) >> p.gs) & ~3;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int off = ((((kbs + j) * SP_BK) + 32 * h) >> p.gs) - c0g;
            cs[h] = W4A16_IN_BOUNDS(off >= 0 && off < p.scb, p.status) ? srow_s[off] : 0.f;
          }
        }
        tc_fence_after();
        if (kbs + j < kb1) {
          uint32_t a[32];
          const uint32_t wv[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint4 d = dequant_word(wv[i], cs[i >> 2], nk_);
            a[4 * i] = d.x; a[4 * i + 1] = d.y; a[4 * i + 2] = d.z; a[4 * i + 3] = d.w;
          }
          tmem_st_32cols(lane_base + SP_A_COL0 + (s * SP_SK + j) * 32, a);
          tmem_store_wait();
        }
        // the words were consumed above: release the weight slot
        __syncwarp();
        if (lane == 0) mbar_arrive(&wempty[ws]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[s]);
      }
    }
    if (ok) {
      // partial tile -> shared memory (the ring is idle once acc_full
      // completes): row r at red[r * SP_RED_LD], 16-byte stores; the padded
      // row stride puts 8 consecutive rows' chunks in 8 different bank groups
      if (j == 0) {
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(acc_full, 0))) {
          fail();
        } else {
          tc_fence_after();
          float *red = reinterpret_cast<float *>(smem) + row * SP_RED_LD;
#pragma unroll 1
          for (int cc = 0; cc < SP_BM / 32; ++cc) {
            uint32_t r[32];
            tmem_ld_32cols(lane_base + cc * 32, r);
#pragma unroll
            for (int t = 0; t < 32; t += 4)
              *reinterpret_cast<uint4 *>(red + cc * 32 + t) =
                  make_uint4(r[t], r[t + 1], r[t + 2], r[t + 3]);
          }
          fence_proxy_async_smem();  // the bulk copies below read the tile
        }
      }
    }
    tc_fence_before();
    __syncwarp();
  }
  __syncthreads();
  // ------------------------------------------------ split-K reduction (push)
  // every rank has parked its partial tile (a failed rank sends whatever
  // its tile holds: the status word already records the failure)
  cluster_wait();  // phase A: every rank's barriers are initialised
  const float *red = reinterpret_cast<const float *>(smem);
  if (threadIdx.x == 0 && ks > 1) push_send<SP_ROWS, SP_RED_LD>(red, recv, red_bar, rank, ks);
  griddep_wait();  // every thread may write y below
  if (ks > 1 && !mbar_wait(red_bar, 0)) fail();
  __syncwarp();
  cluster_arrive();  // phase B: the slices of this rank's rows have landed
  if (*reinterpret_cast<volatile int *>(abort_flag) == 0)
    push_owner_sum<SP_ROWS, SP_BM, SP_RED_LD, SP_MAX_KS>(red, recv, rank, ks, n0, m0, p.M, p.N,
                                                         p.y, p.ybf16, p.status);
  cluster_wait();  // phase B: every slice this CTA sent has landed
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(SP_TMEM_COLS)
                 : "memory");
  }
}

}  // namespace

cudaError_t launch_tc_split(const uint16_t *x, const int32_t *qw, const float *sc, int M, int N,
                            int K, int group, void *y, bool y_bf16, bool overlap, int kmax,
                            cudaStream_t stream) {
  const DeviceInfo &di = device_info();
  auto encode = encode_fn();
  if (encode == nullptr) return cudaErrorNotSupported;
  CUtensorMap tmap;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
  const cuuint32_t box[2] = {SP_BK, SP_BM};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(x), dims,
                      strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  // packed weights [N][K/8] words: one 32-word (128-byte) x 128-row box per
  // stage, 128-byte swizzle, zeros past K and N
  CUtensorMap tmap_w;
  const cuuint64_t wdims[2] = {static_cast<cuuint64_t>(K / 8), static_cast<cuuint64_t>(N)};
  const cuuint64_t wstrides[1] = {static_cast<cuuint64_t>(K / 8) * 4};
  const cuuint32_t wbox[2] = {SP_SK * 8, SP_ROWS};
  r = encode(&tmap_w, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<int32_t *>(qw), wdims, wstrides,
             wbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  SpParams p{};
  p.qw = qw;
  p.sc = sc;
  p.y = y;
  p.ybf16 = y_bf16 ? 1 : 0;
  p.M = M;
  p.N = N;
  p.K = K;
  p.gs = group == 128 ? 7 : group == 64 ? 6 : 5;
  p.scb = group == 32 ? 8 : 4;
  p.status = di.status;
  // scales [N][K/group] fp32 by TMA when a scale row is a whole number of
  // 16-byte units: a box of scb floats x 128 rows per stage, zeros past the
  // row's end and past N (an aligned window of 4 groups holds a stage's 2
  // groups of 128 columns; with groups of 32 a stage starts on a multiple
  // of 8 groups, with 64 on a multiple of 4)
  const int G = K / group;
  const bool sct = G % 4 == 0 && (reinterpret_cast<uintptr_t>(sc) & 15u) == 0;
  CUtensorMap tmap_s = tmap_w;
  if (sct) {
    const cuuint64_t sdims[2] = {static_cast<cuuint64_t>(G), static_cast<cuuint64_t>(N)};
    const cuuint64_t sstrides[1] = {static_cast<cuuint64_t>(G) * 4};
    const cuuint32_t sbox[2] = {static_cast<cuuint32_t>(p.scb), SP_ROWS};
    r = encode(&tmap_s, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(sc), sdims, sstrides,
               sbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  const int tiles_m = (M + SP_BM - 1) / SP_BM;
  const int tiles_n = (N + SP_ROWS - 1) / SP_ROWS;
  // split K over a cluster of up to kmax CTAs (a power of two, at most the
  // number of stages) so that the clusters cover the SMs once
  const int nst = (K + SP_BK * SP_SK - 1) / (SP_BK * SP_SK);
  int lks = 0;
  while ((2 << lks) <= std::min(std::min(std::min(kmax, SP_MAX_KS), nst),
                                di.num_sms / std::max(1, tiles_m * tiles_n)))
    ++lks;
  p.lks = lks;

  auto kern = sct ? tc_split_kernel<true> : tc_split_kernel<false>;
  static PerDeviceOnce attr_once[2];
  const cudaError_t attr_err = attr_once[sct ? 1 : 0].run(
      [&] { return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SP_SMEM); });
  if (attr_err != cudaSuccess) return attr_err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles_n, 1 << lks, tiles_m);
  cfg.blockDim = dim3(SP_THREADS);
  cfg.dynamicSmemBytes = SP_SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = 1 << lks;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = overlap ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, tmap, tmap_w, tmap_s, p);
}

}  // namespace w4a16
