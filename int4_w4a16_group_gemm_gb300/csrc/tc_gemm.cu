// Large-M W4A16 GEMM on the 5th-generation (tcgen05) tensor cores, bf16
// activations, fp32 accumulation in tensor memory.
//
//   y[m][n] = sum_k x[m][k] * W_hat[n][k],  W_hat = (nibble - 8) * scale
//
// The contraction is computed transposed, D[n][m] = W_hat_tile * x_tile^T,
// so that the dequantised weights are the MMA's A operand (M = 128 weight
// rows per instruction) and the activations its B operand (N = 256 token
// rows). One CTA owns a 256 (weights) x 256 (tokens) output tile: two
// 128-row A sub-tiles share every B tile, each with its own 256-column fp32
// accumulator, filling all 512 TMEM columns.
//
// Warp roles (320 threads, one CTA per SM, persistent over tiles):
//   warp 0      TMA producer: 2-D tiled loads of x (128-byte swizzle) into
//               the B slot and of the packed words into the W slot of each
//               pipeline stage;
//   warp 1      TMEM owner and MMA issuer: the warp runs the issue loop
//               and one elected lane issues tcgen05.mma (kind::f16, bf16 x
//               bf16 -> f32) per 16-wide K step and commits each stage back
//               to its producers;
//   warps 2-9   dequantisers: thread r owns weight row r of the tile, reads
//               its packed words from the stage (TMA) and loads its scales
//               from global memory two stages ahead, forms fp32
//               (nibble - 8) * scale exactly, rounds to bf16 and stores the
//               16-byte chunks in the canonical K-major 128-byte swizzled
//               layout the MMA reads; after a tile's last stage the same
//               warps drain the accumulators (tcgen05.ld) to y.
// Stage = 64 K columns: A 2 x 16 KB (dequantised) + B 32 KB (TMA) + the
// packed words 8 KB (TMA, one 8-word x 256-row box); 3 stages.
// Every wait is bounded; a timeout is recorded in the status word and the
// CTA unwinds (TMEM is always freed).
//
// Format: "The Quiet Commit: How a Single Documentation Edit Marks the
// Completion of a Major Engineering Milestone", section "The INT4 Milestone".
// The pages' kernel ran on CUDA cores for sm_120; tensor cores are used here
// because at large M the product is a dense contraction.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdlib>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "tc_core.cuh"

namespace w4a16 {

namespace {

using namespace tc;

constexpr int TC_BK = 64;   // K per stage: one 128-byte swizzle row of bf16
constexpr int A_SUB_BYTES = 128 * TC_BK * 2;        // 16 KB

// Tile shape. BM is the token width (the MMA N); SUBS the number of
// 128-row weight sub-tiles per CTA (each an MMA M = 128 with its own TMEM
// accumulator of BM columns): BM = 256, SUBS = 2. (Small M runs on the
// split-K kernel of tc_split.cu.)
template <int BM, int SUBS>
struct TcCfg {
  static constexpr int kDqWarps = 8;                        // dequantiser warps
  static constexpr int kThreads = 64 + 32 * kDqWarps;      // + TMA warp + MMA warp
  static constexpr int kRows = 128 * SUBS;                 // weight rows per tile
  static constexpr int kABytes = SUBS * A_SUB_BYTES;
  static constexpr int kBBytes = BM * TC_BK * 2;
  static constexpr int kWBytes = kRows * TC_BK / 2;  // the stage's packed words (TMA)
  static constexpr int kStageBytes = kABytes + kBBytes + kWBytes;
  static constexpr int kBlocks = 3;   // 64-column blocks in the ring
  // blocks per pipeline stage (one barrier handshake per stage); a stage of
  // this tile already carries 16 MMAs of N = 256
  static constexpr int kSubK = 1;
  static constexpr int kStages = kBlocks / kSubK;
  static constexpr int kPrefetch = 2;  // stages of scales in flight per thread
  static constexpr int kThreadsPerRow = 32 * kDqWarps / kRows;  // dequant threads per row
  static constexpr int kTmemCols = SUBS * BM < 32 ? 32 : SUBS * BM;  // a power of two
  static constexpr int kSmem = kBlocks * kStageBytes + 1024 + 256;
  static_assert(kSubK == 1, "one 64-column block per stage (one packed-word box)");
  static_assert(kSmem <= 227 * 1024, "shared memory");
  // Instruction descriptor, kind::f16: D f32 (bits 4-5 = 1), A bf16 (bits
  // 7-9 = 1), B bf16 (bits 10-12 = 1), both K-major (bits 15, 16 = 0),
  // N >> 3 in bits 17-22, M >> 4 in bits 24-28.
  static constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) |
                                     (static_cast<uint32_t>(BM >> 3) << 17) |
                                     (static_cast<uint32_t>(128 >> 4) << 24);
};

struct TcParams {
  const int32_t *qw;
  const float *sc;
  void *y;  // fp32, or bf16 when ybf16
  int ybf16;
  int M, N, K;
  int tiles_m, num_tiles;
  int gs;  // log2 of the group size
  int *status;
};

// Persistent CTAs walk the (weight-tile, token-tile) grid, each tile over
// all of K.
template <int BM, int SUBS>
__global__ void __launch_bounds__(TcCfg<BM, SUBS>::kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmap_x,
                   const __grid_constant__ CUtensorMap tmap_w, const TcParams p) {
  using Cfg = TcCfg<BM, SUBS>;
  constexpr int NS = Cfg::kStages;
  constexpr int SK = Cfg::kSubK;       // 64-column blocks per stage
  constexpr int SB = Cfg::kStageBytes;  // bytes of one block (A then B)
  constexpr int PD = Cfg::kPrefetch;
  constexpr int ROWS = Cfg::kRows;
  constexpr int TPR = Cfg::kThreadsPerRow;
  constexpr int WPT = 8 / TPR;  // packed words per dequant thread per stage
  constexpr int DQ_WARPS = Cfg::kDqWarps;
  constexpr int PIECES = WPT >= 4 ? WPT / 4 : 1;  // 16-byte loads per stage
  constexpr int PW = WPT >= 4 ? 4 : WPT;          // words per load
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + NS * SK * SB);
  uint64_t *empty = full + NS;
  uint64_t *wfull = empty + NS;  // [NS] the stage's packed words have landed
  uint64_t *acc_full = wfull + NS;
  uint64_t *acc_empty = acc_full + 1;
  uint64_t *drain = acc_empty + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = p.K;
  const int nk = (K + TC_BK - 1) / TC_BK;
  const int kb0 = 0, kb1 = nk;  // every tile covers all of K
  const int tile_first = blockIdx.x;
  const int tile_step = gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1 + DQ_WARPS);
      mbar_init(&empty[s], 1);
      mbar_init(&wfull[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, DQ_WARPS);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(Cfg::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Programmatic launch: let the next kernel on the stream start launching
  // now. Only the weights (never written by the previous kernel, by the
  // overlap contract) are read before griddep_wait; x and y after it. Both
  // calls are no-ops for a kernel launched without the attribute.
  griddep_launch_dependents();

  auto fail = [&]() {
    record_status(p.status, W4A16_ERR_TIMEOUT);
    *reinterpret_cast<volatile int *>(abort_flag) = 1;
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA
    if (lane == 0) {
      griddep_wait();
      // the activation tiles are re-read by every weight tile of their token
      // tile, in later waves too: keep them in L2 ahead of the weights and
      // the output stream
      const uint64_t keep = l2_policy_evict_last();
      int it = 0;
      for (int tile = tile_first; tile < p.num_tiles && !aborted(abort_flag); tile += tile_step) {
        const int m0 = (tile % p.tiles_m) * BM;
        const int n0 = (tile / p.tiles_m) * ROWS;
        for (int kb = kb0; kb < kb1; kb += SK, ++it) {
          const int s = it % NS;
          const uint32_t ph = static_cast<uint32_t>(it / NS) & 1u;
          if (!mbar_wait(&empty[s], ph ^ 1u)) { fail(); break; }
          if (aborted(abort_flag)) break;
          uint8_t *st = smem + s * SB;
          // the packed words of the tile's rows (one 8-word x ROWS box, zeros
          // past K and N), then the activation tile
          mbar_arrive_expect_tx(&wfull[s], static_cast<uint32_t>(Cfg::kWBytes));
          tma_load_2d(st + Cfg::kABytes + Cfg::kBBytes, &tmap_w, kb * 8, n0, &wfull[s]);
          mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(Cfg::kBBytes));
          tma_load_2d_hint(st + Cfg::kABytes, &tmap_x, kb * TC_BK, m0, &full[s], keep);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
    // the whole warp runs this loop (warp-uniform operands); one elected
    // lane issues (tc_mma_warp); waits are taken by lane 0 and broadcast
    int it = 0, tcount = 0;
    bool issued_any = false;
    for (int tile = tile_first; tile < p.num_tiles; tile += tile_step, ++tcount) {
      int st = 0;  // 1: another warp failed, 2: this wait timed out
      if (lane == 0) {
        if (aborted(abort_flag)) st = 1;
        else if (tcount > 0 && !mbar_wait(acc_empty, static_cast<uint32_t>(tcount - 1) & 1u)) st = 2;
      }
      st = __shfl_sync(0xFFFFFFFFu, st, 0);
      if (st == 2 && lane == 0) fail();
      if (st != 0) break;
      tc_fence_after();
      bool ok = true;
      for (int kb = kb0; kb < kb1; kb += SK, ++it) {
        const int s = it % NS;
        const uint32_t ph = static_cast<uint32_t>(it / NS) & 1u;
        const int nsub = min(SK, kb1 - kb);
        int got = 1;
        if (lane == 0) got = mbar_wait(&full[s], ph) && !aborted(abort_flag);
        if (!__shfl_sync(0xFFFFFFFFu, got, 0)) {
          if (lane == 0) fail();
          ok = false;
          break;
        }
        tc_fence_after();
        for (int j = 0; j < nsub; ++j) {
          const uint32_t a0 = smem_u32(smem + (s * SK + j) * SB);
          const uint64_t ad = sw128_desc(a0), bd = sw128_desc(a0 + Cfg::kABytes);
#pragma unroll
          for (int sub = 0; sub < SUBS; ++sub)
#pragma unroll
            for (int k = 0; k < TC_BK / 16; ++k)  // +32 bytes per K step: +2 in the start field
              tc_mma_warp(tmem + sub * BM, ad + sub * (A_SUB_BYTES >> 4) + 2 * k, bd + 2 * k,
                          Cfg::kIdesc, (kb + j > kb0 || k > 0) ? 1u : 0u);
        }
        tc_commit_warp(&empty[s]);
        issued_any = true;
      }
      if (!ok) break;
      tc_commit_warp(acc_full);
    }
    // all MMAs this warp issued are complete before TMEM is released
    if (issued_any) {
      tc_commit_warp(drain);
      if (lane == 0) mbar_wait(drain, 0);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------- dequant + epilogue
    const NibbleConsts nk = make_nibble_consts();
    const int dq = threadIdx.x - 64;                  // 0 .. 32 * DQ_WARPS - 1
    const int row = dq / TPR, part = dq % TPR;        // weight row within the tile
    const int sub = row >> 7, rr = row & 127;
    const int Kw = K >> 3;                            // packed words per row
    const int G = K >> p.gs;
    // this row's byte offset inside the A region (swizzle applied per chunk)
    const uint32_t row_off =
        static_cast<uint32_t>(sub * A_SUB_BYTES + (rr >> 3) * 1024 + (rr & 7) * 128);
    const int swz = rr & 7;
    // this thread's words inside a stage's packed-word box
    (void)W4A16_IN_BOUNDS(row * (TC_BK / 2) + (part + 1) * WPT * 4 <= Cfg::kWBytes, p.status);
    const int q = warp & 3;                  // TMEM lane quadrant of this warp
    const int esub = (warp - 2) >> 2;        // accumulator this warp drains
    int it = 0, tcount = 0;
    for (int tile = tile_first; tile < p.num_tiles && !aborted(abort_flag);
         tile += tile_step, ++tcount) {
      const int n0 = (tile / p.tiles_m) * ROWS;
      const int m0 = (tile % p.tiles_m) * BM;
      const int n = n0 + row;
      const bool nvalid = n < p.N;
      const float *srow = p.sc + static_cast<size_t>(n) * G;

      // register ring of PD prefetched stages of scales (slots indexed at
      // compile time); the packed words come by TMA with the stage
      float rs[PD][SK][PIECES];
      auto fetch = [&](int kb, float (&sc)[PIECES]) {
#pragma unroll
        for (int h = 0; h < PIECES; ++h) sc[h] = 0.f;
        if (!nvalid || kb >= kb1) return;
#pragma unroll
        for (int h = 0; h < PIECES; ++h) {
          const int w0 = kb * 8 + part * WPT + PW * h;  // first word of this piece
          // a piece past K keeps scale 0 (its zero-filled words then weigh 0)
          if (w0 < Kw && W4A16_IN_BOUNDS(n < p.N && w0 + PW <= Kw && ((w0 * 8) >> p.gs) < G,
                                         p.status))
            sc[h] = __ldg(srow + ((w0 * 8) >> p.gs));  // a piece lies in one group
        }
      };
#pragma unroll
      for (int u = 0; u < PD; ++u)
#pragma unroll
        for (int j = 0; j < SK; ++j) fetch(kb0 + u * SK + j, rs[u][j]);
      bool ok = true;
      // one stage (SK blocks) per iteration: the SK blocks' words are
      // independent, so their dequantisation interleaves
      for (int kbase = kb0; kbase < kb1 && ok; kbase += PD * SK) {
#pragma unroll
        for (int u = 0; u < PD; ++u) {
          const int kbs = kbase + u * SK;  // first block of the stage
          if (kbs >= kb1) break;
          const int nsub = min(SK, kb1 - kbs);
          const int s = it % NS;
          const uint32_t ph = static_cast<uint32_t>(it / NS) & 1u;
          ++it;
          float cs[SK][PIECES];
#pragma unroll
          for (int j = 0; j < SK; ++j)
#pragma unroll
            for (int h = 0; h < PIECES; ++h) cs[j][h] = rs[u][j][h];
#pragma unroll
          for (int j = 0; j < SK; ++j) fetch(kbs + PD * SK + j, rs[u][j]);
          // the stage's packed words have landed (the producer loads them
          // once the stage's previous MMAs are complete, so its A region is
          // free too)
          const bool got =
              __all_sync(0xFFFFFFFFu, mbar_wait(&wfull[s], ph) && !aborted(abort_flag));
          if (!got) { fail(); ok = false; break; }
          uint32_t cw[SK][WPT];
#pragma unroll
          for (int j = 0; j < SK; ++j) {
            const uint8_t *wrow = smem + (s * SK + j) * SB + Cfg::kABytes + Cfg::kBBytes +
                                  row * (TC_BK / 2) + part * WPT * 4;
#pragma unroll
            for (int h = 0; h < PIECES; ++h) {
              if (PW == 4) {
                const uint4 v = *reinterpret_cast<const uint4 *>(wrow + 16 * h);
                cw[j][4 * h] = v.x; cw[j][4 * h + 1] = v.y; cw[j][4 * h + 2] = v.z;
                cw[j][4 * h + 3] = v.w;
              } else {
#pragma unroll
                for (int i = 0; i < PW; ++i)
                  cw[j][PW * h + i] = reinterpret_cast<const uint32_t *>(wrow)[PW * h + i];
              }
            }
          }
#pragma unroll
          for (int j = 0; j < SK; ++j) {
            if (j < nsub) {
              uint8_t *arow = smem + (s * SK + j) * SB + row_off;
              // this row's 128 bytes of the stage's A region
              (void)W4A16_IN_BOUNDS(row_off + 128u <= static_cast<uint32_t>(Cfg::kABytes), p.status);
#pragma unroll
              for (int i = 0; i < WPT; ++i) {
                const int chunk = part * WPT + i;
                *reinterpret_cast<uint4 *>(arow + ((chunk ^ swz) << 4)) =
                    dequant_word(cw[j][i], cs[j][i / PW], nk);
              }
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&full[s]);
        }
      }
      if (!ok) break;
      griddep_wait();  // before the first write of y
      // -------- epilogue: accumulator esub, TMEM lanes q*32 .. q*32+31
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(acc_full, static_cast<uint32_t>(tcount) & 1u))) {
        fail();
        break;
      }
      tc_fence_after();
      if (esub < SUBS) {
        const int nl = esub * 128 + q * 32 + lane;  // row within the tile
        const int ne = n0 + nl;
        const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16) + esub * BM;
#pragma unroll 1
        for (int cc = 0; cc < BM / 32; ++cc) {
          uint32_t r[32];
          tmem_ld_32cols(tbase + cc * 32, r);
          const int mb = m0 + cc * 32;
          if (ne < p.N) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (mb + j < p.M && W4A16_IN_BOUNDS(ne >= 0 && ne < p.N, p.status))
                store_y(p.y, static_cast<size_t>(mb + j) * p.N + ne, __uint_as_float(r[j]),
                        p.ybf16);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty);
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(Cfg::kTmemCols)
                 : "memory");
  }
}

}  // namespace

bool tc_gemm_supported(int M, int N, int K) {
  return M > 0 && N > 0 && K > 0 && K % 32 == 0;
}

namespace {

template <int BM, int SUBS>
cudaError_t launch_tc(const CUtensorMap &tmap, const CUtensorMap &tmap_w, const TcParams &p,
                      int grid_x, bool overlap, cudaStream_t stream) {
  using Cfg = TcCfg<BM, SUBS>;
  auto kern = tc_gemm_kernel<BM, SUBS>;
  static PerDeviceOnce attr_once;
  const cudaError_t attr_err = attr_once.run([&] {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
  });
  if (attr_err != cudaSuccess) return attr_err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid_x);
  cfg.blockDim = dim3(Cfg::kThreads);
  cfg.dynamicSmemBytes = Cfg::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = overlap ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tmap, tmap_w, p);
}

int env_int(const char *name) {
  const char *v = getenv(name);
  return v ? atoi(v) : 0;
}

}  // namespace

cudaError_t launch_tc_gemm(const uint16_t *x, const int32_t *qw, const float *sc, int M, int N,
                           int K, int group, void *y, bool y_bf16, bool overlap,
                           cudaStream_t stream) {
  const DeviceInfo &di = device_info();
  // 128 x 64 tiles with K split over a cluster (tc_split.cu) for M <= 64,
  // and for larger M while those tiles fit in one wave (measured at
  // K = 7168: a one-wave split launch beats the persistent kernel up to
  // M = 512); otherwise 256 x 256 persistent tiles here.
  static const int env_variant = env_int("W4A16_TC_VARIANT");  // tuning override
  const long long split_tiles = static_cast<long long>((M + 63) / 64) * ((N + 127) / 128);
  bool small = M <= 64 || split_tiles <= di.num_sms;
  if (env_variant == 1) small = true;
  if (env_variant == 2) small = false;
  if (small) {
    static const int env_ks = env_int("W4A16_TC_KS");  // tuning override
    const int kmax = env_ks > 0 ? std::min(env_ks, 8) : 4;
    return launch_tc_split(x, qw, sc, M, N, K, group, y, y_bf16, overlap, kmax, stream);
  }
  auto encode = encode_fn();
  if (encode == nullptr) return cudaErrorNotSupported;
  constexpr int BM = 256, ROWS = 256;
  CUtensorMap tmap;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
  const cuuint32_t box[2] = {TC_BK, static_cast<cuuint32_t>(BM)};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(x), dims,
                      strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  // packed words [N][K/8]: 8 words (one 64-column block) x ROWS rows per box,
  // zeros past K and N
  CUtensorMap tmap_w;
  const cuuint64_t wdims[2] = {static_cast<cuuint64_t>(K / 8), static_cast<cuuint64_t>(N)};
  const cuuint64_t wstrides[1] = {static_cast<cuuint64_t>(K / 8) * 4};
  const cuuint32_t wbox[2] = {TC_BK / 8, static_cast<cuuint32_t>(ROWS)};
  r = encode(&tmap_w, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<int32_t *>(qw), wdims,
             wstrides, wbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  TcParams p{};
  p.qw = qw;
  p.sc = sc;
  p.y = y;
  p.ybf16 = y_bf16 ? 1 : 0;
  p.M = M;
  p.N = N;
  p.K = K;
  p.tiles_m = (M + BM - 1) / BM;
  p.num_tiles = p.tiles_m * ((N + ROWS - 1) / ROWS);
  p.gs = group == 128 ? 7 : group == 64 ? 6 : 5;
  p.status = di.status;
  return launch_tc<BM, 2>(tmap, tmap_w, p, std::min(p.num_tiles, di.num_sms), overlap, stream);
}

}  // namespace w4a16
