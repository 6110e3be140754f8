// Small-M W4A16 GEMM with fp32 activations on the tcgen05 tensor cores,
// exact to fp32 accumulation:
//
//   y[m][n] = sum_g sc[n][g] * D_g[n][m],   D_g[n][m] = sum_{k in g} (nib[n][k] - 8) * x[m][k]
//
// Two exact splits make the contraction a bf16 one:
//   * every fp32 activation is the sum of three bf16 numbers,
//     x = x1 + x2 + x3 with x1 = bf16(x), x2 = bf16(x - x1), x3 = x - x1 - x2
//     (each difference is exact in fp32, and 24 significant bits fit in
//     three 8-bit pieces);
//   * (nib - 8) is a small integer, exact in bf16.
// The products (nib - 8) * x_i are exact, the tensor cores add them in fp32
// into TMEM, one 32-column group at a time: per 16 columns one MMA of N = 64
// for each piece, all three into the group's accumulator, in a ring of six
// accumulators (so the MMAs run up to five groups ahead of the readback);
// readback warps multiply each group's sum by its fp32 scale and accumulate
// in registers. The scale never passes through bf16, so the result carries
// only fp32 summation error. The depth per output is the 6 MMAs of a
// 32-column group inside the tensor core, the CTA's groups (an fp32 FMA
// chain, at most 128 for K <= 16384), then the split-K partials of the
// cluster in rank order.
//
// Tile: 128 weight rows x 64 tokens; K is split over a cluster of up to 4
// CTAs exactly as in the bf16 small-M kernel, whose cluster reduction this
// kernel reuses. Stage = 64 columns (two groups):
//   A   (nib - 8) in bf16, 128 TMEM lanes x 32 columns (tcgen05.st by the
//       dequantisers; the MMAs read A from tensor memory, so it costs no
//       shared-memory bandwidth)
//   B   3 x 8 KB  the activation pieces, canonical K-major 128-byte swizzle
// in a ring of 4 MMA stages, and the fp32 activation tiles (16 KB, loaded
// by TMA as two 128-byte-swizzled halves) in a separate ring of 3 that the
// dequantisers release as soon as they have split a tile, so activation
// loads run ahead of the MMAs.
// Within every 8-column word the K order of A and B is (0,4,1,5,2,6,3,7):
// the bf16 magic-number unpack yields nibbles c and c+4 together, and a
// contraction is unchanged by one permutation of K applied to both operands.
//
// Warp roles (448 threads, one CTA per SM):
//   warp 0       TMA of the fp32 activation tiles;
//   warp 1       TMEM owner and MMA issuer;
//   warps 2-9    dequantisers: (nib - 8) tiles of A (warp w: TMEM lane
//                quadrant w % 4, half (w - 2) / 4 of each stage's words)
//                and the three pieces of B;
//   warps 10-13  readback: TMEM lanes of one quadrant each, scale, accumulate,
//                and at the end the partial tile for the cluster reduction.
// Every wait is bounded; a timeout is recorded and the CTA unwinds.
//
// Format: "The Quiet Commit: How a Single Documentation Edit Marks the
// Completion of a Major Engineering Milestone", section "The INT4 Milestone"
// (fp32 activations, INT4 weights, fp32 group scales); fp32 accumulation:
// "The Silence of Success: A Single Line That Speaks Volumes", section
// "Assumptions Embedded in the Code".
#include <algorithm>
#include <cstdlib>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "tc_core.cuh"

namespace w4a16 {

namespace {

using namespace tc;

constexpr int FX_BK = 64;          // K columns per stage (two groups)
constexpr int FX_BM = 64;          // tokens per tile (the MMA N)
constexpr int FX_ROWS = 128;       // weight rows per tile (the MMA M)
constexpr int FX_DQ_WARPS = 8;
constexpr int FX_RB_WARPS = 4;
constexpr int FX_THREADS = 64 + 32 * (FX_DQ_WARPS + FX_RB_WARPS);
constexpr int FX_B_BYTES = FX_BM * FX_BK * 2;    // 8 KB per piece
constexpr int FX_X_BYTES = FX_BM * FX_BK * 4;    // 16 KB
constexpr int FX_STAGE = 3 * FX_B_BYTES;        // one MMA stage in shared memory (B)
constexpr int FX_NS = 4;            // MMA stages
constexpr int FX_NSX = 3;           // fp32 activation tiles in flight
constexpr int FX_PD = 2;            // stages of packed weights prefetched per thread
constexpr int FX_NB = FX_BM;        // MMA N: the tile's tokens
constexpr int FX_ACC = 6;           // group accumulators in TMEM (FX_NB columns each)
constexpr int FX_TMEM_COLS = 512;   // the accumulators, then the A ring
constexpr int FX_A_COL0 = FX_ACC * FX_NB;  // A stage s at column FX_A_COL0 + 32 s
static_assert(FX_A_COL0 + FX_NS * 32 <= FX_TMEM_COLS, "TMEM budget");
constexpr int FX_RED_LD = FX_BM + 4;  // row stride of the parked partial tile (floats)
constexpr int FX_MAX_KS = 4;          // largest cluster (K split)
constexpr int FX_RECV_BYTES = push_recv_bytes<FX_ROWS, FX_RED_LD, FX_MAX_KS>();
constexpr int FX_SMEM = FX_NS * FX_STAGE + FX_NSX * FX_X_BYTES + FX_RECV_BYTES + 1024 + 256;
static_assert(FX_ROWS * FX_RED_LD * 4 <= FX_NS * FX_STAGE, "parked partial tile");
// Instruction descriptor, kind::f16: D f32, A and B bf16, both K-major,
// N = 64 (one piece tile), M = 128.
constexpr uint32_t FX_IDESC = (1u << 4) | (1u << 7) | (1u << 10) |
                              (static_cast<uint32_t>(FX_NB >> 3) << 17) |
                              (static_cast<uint32_t>(FX_ROWS >> 4) << 24);

struct FxParams {
  const int32_t *qw;
  const float *sc;
  void *y;  // fp32, or bf16 when ybf16
  int ybf16;
  int M, N, K;
  int num_tiles;
  int gs;  // log2 of the group size
  int *status;
};

// The packed word of 8 nibbles as four bf16x2 pairs (n_c - 8, n_{c+4} - 8),
// c = 0..3, in a uint4: 128 + n is an exact bf16 (the pattern 0x4300 ORs n
// into the mantissa), and one bf16x2 subtraction of 136 leaves n - 8.
__device__ __forceinline__ uint4 dequant_word_int(uint32_t w, uint32_t magic, uint32_t bias) {
  uint32_t p[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint32_t h = ((w >> (4 * c)) & 0x000F000Fu) | magic;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(p[c]) : "r"(h), "r"(bias));
  }
  return make_uint4(p[0], p[1], p[2], p[3]);
}

// Eight fp32 activations (columns 0..7 of a word) -> three bf16 chunks
// x1, x2, x3 with x = x1 + x2 + x3 exactly, each chunk in the K order
// (0,4,1,5,2,6,3,7).
__device__ __forceinline__ void split_chunk(const float (&v)[8], uint4 &o1, uint4 &o2, uint4 &o3) {
  uint32_t a[4], b[4], c[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float lo = v[j], hi = v[j + 4];
    a[j] = pack_bf16x2(lo, hi);
    const float r1l = lo - __uint_as_float(a[j] << 16);
    const float r1h = hi - __uint_as_float(a[j] & 0xFFFF0000u);
    b[j] = pack_bf16x2(r1l, r1h);
    const float r2l = r1l - __uint_as_float(b[j] << 16);
    const float r2h = r1h - __uint_as_float(b[j] & 0xFFFF0000u);
    c[j] = pack_bf16x2(r2l, r2h);
  }
  o1 = make_uint4(a[0], a[1], a[2], a[3]);
  o2 = make_uint4(b[0], b[1], b[2], b[3]);
  o3 = make_uint4(c[0], c[1], c[2], c[3]);
}

// Byte offset of 16-byte chunk `chunk` of row `row` in a K-major tile with
// 128-byte swizzle (8-row atoms of 1024 bytes).
__device__ __forceinline__ uint32_t sw128_offset(int row, int chunk) {
  return static_cast<uint32_t>((row >> 3) * 1024 + (row & 7) * 128 + ((chunk ^ (row & 7)) << 4));
}

__global__ void __launch_bounds__(FX_THREADS, 1)
    tc_f32_kernel(const __grid_constant__ CUtensorMap tmap_x, const FxParams p) {
  constexpr int NS = FX_NS;
  constexpr int SB = FX_STAGE;
  constexpr int PD = FX_PD;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *xring = smem + NS * SB;                                 // fp32 activation tiles
  float *recv = reinterpret_cast<float *>(xring + FX_NSX * FX_X_BYTES);  // split-K slices
  uint64_t *full = reinterpret_cast<uint64_t *>(xring + FX_NSX * FX_X_BYTES + FX_RECV_BYTES);
  uint64_t *xfull = full + NS;                                     // [FX_NSX] tile landed
  uint64_t *xempty = xfull + FX_NSX;                               // [FX_NSX] tile split
  uint64_t *empty = xempty + FX_NSX;                               // MMAs of the stage done
  uint64_t *acc_full = empty + NS;                                 // [FX_ACC] group sum ready
  uint64_t *acc_empty = acc_full + FX_ACC;                         // [FX_ACC] group sum read
  uint64_t *drain = acc_empty + FX_ACC;
  uint64_t *red_bar = drain + 1;  // split-K slices of this rank's rows landed
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(red_bar + 1);
  int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = p.K;
  const int Kw = K >> 3;
  const int G32 = K >> 5;       // 32-column groups (the MMA's unit)
  const int G = K >> p.gs;       // scale groups per row
  const int gsh = p.gs - 5;      // 32-column groups per scale group, log2
  const int nk = (K + FX_BK - 1) / FX_BK;
  const int rank = static_cast<int>(blockIdx.y);
  const int ks = static_cast<int>(gridDim.y);
  const int kb0 = static_cast<int>((static_cast<long long>(nk) * rank) / ks);
  const int kb1 = static_cast<int>((static_cast<long long>(nk) * (rank + 1)) / ks);
  const int tile = blockIdx.x;
  const int n0 = tile * FX_ROWS;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], FX_DQ_WARPS);
      mbar_init(&empty[s], 1);
    }
    for (int x = 0; x < FX_NSX; ++x) {
      mbar_init(&xfull[x], 1);
      mbar_init(&xempty[x], FX_DQ_WARPS);
    }
    for (int b = 0; b < FX_ACC; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], FX_RB_WARPS);
    }
    mbar_init(drain, 1);
    mbar_init(red_bar, 1);
    if (ks > 1) push_expect<FX_ROWS, FX_RED_LD>(red_bar, ks);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(FX_TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_arrive();  // phase A: this rank's barriers are initialised
  const uint32_t tmem = *tmem_slot;
  // Programmatic launch: the weights are read before griddep_wait, x and y
  // after it (no-ops without the launch attribute).
  griddep_launch_dependents();

  auto fail = [&]() {
    record_status(p.status, W4A16_ERR_TIMEOUT);
    *reinterpret_cast<volatile int *>(abort_flag) = 1;
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA
    if (lane == 0) {
      griddep_wait();
      for (int kb = kb0, it = 0; kb < kb1 && !aborted(abort_flag); ++kb, ++it) {
        const int x = it % FX_NSX;
        const uint32_t ph = static_cast<uint32_t>(it / FX_NSX) & 1u;
        if (!mbar_wait(&xempty[x], ph ^ 1u)) { fail(); break; }
        mbar_arrive_expect_tx(&xfull[x], FX_X_BYTES);
        // two 32-column boxes (128-byte rows, 128-byte swizzle)
        tma_load_2d(xring + x * FX_X_BYTES, &tmap_x, kb * FX_BK, 0, &xfull[x]);
        tma_load_2d(xring + x * FX_X_BYTES + FX_X_BYTES / 2, &tmap_x, kb * FX_BK + 32, 0,
                    &xfull[x]);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
    // the whole warp runs this loop (warp-uniform operands); one elected
    // lane issues (tc_mma_tmem_a_warp); waits are taken by lane 0 and
    // broadcast
    int g = 0;  // group counter: buffer g % FX_ACC, use g / FX_ACC
    bool issued_any = false;
    for (int kb = kb0, it = 0; kb < kb1; ++kb, ++it) {
      const int s = it % NS;
      const uint32_t ph = static_cast<uint32_t>(it / NS) & 1u;
      int got = 1;
      if (lane == 0) got = mbar_wait(&full[s], ph) && !aborted(abort_flag);
      if (!__shfl_sync(0xFFFFFFFFu, got, 0)) {
        if (lane == 0) fail();
        break;
      }
      tc_fence_after();
      const uint32_t a0 = tmem + FX_A_COL0 + s * 32;  // (nib - 8) in TMEM
      const uint64_t b0 = sw128_desc(smem_u32(smem + s * SB));
      const int groups = min(2, G32 - 2 * kb);  // the last stage may hold one group
      bool ok = true;
      for (int h = 0; h < groups; ++h, ++g) {
        const int buf = g % FX_ACC;
        int free_ = 1;
        if (lane == 0)
          free_ = mbar_wait(&acc_empty[buf], (static_cast<uint32_t>(g / FX_ACC) & 1u) ^ 1u) &&
                  !aborted(abort_flag);
        if (!__shfl_sync(0xFFFFFFFFu, free_, 0)) {
          if (lane == 0) fail();
          ok = false;
          break;
        }
        tc_fence_after();
        // the three pieces' products go into the same accumulator (piece
        // tile p starts FX_B_BYTES / 16 units further in the start field)
#pragma unroll
        for (int pc = 0; pc < 3; ++pc)
#pragma unroll
          for (int k = 0; k < 2; ++k)  // +32 bytes per K step: +2 in the start field
            tc_mma_tmem_a_warp(tmem + buf * FX_NB, a0 + (2 * h + k) * 8,
                               b0 + pc * (FX_B_BYTES >> 4) + 2 * (2 * h + k), FX_IDESC,
                               (pc > 0 || k > 0) ? 1u : 0u);
        tc_commit_warp(&acc_full[buf]);
        issued_any = true;
      }
      if (!ok) break;
      tc_commit_warp(&empty[s]);
    }
    // every MMA this warp issued is complete before TMEM is released
    if (issued_any) {
      tc_commit_warp(drain);
      if (lane == 0) mbar_wait(drain, 0);
    }
    __syncwarp();
  } else if (warp < 2 + FX_DQ_WARPS) {
    // -------------------------------------------------------- dequantisers
    const uint32_t magic = opaque_u32(0x43004300u);  // bf16 pair (128, 128)
    const uint32_t bias = opaque_u32(0x43084308u);   // bf16 pair (136, 136)
    const int dq = threadIdx.x - 64;                  // 0 .. 255
    // A: TMEM lane = weight row; warp w may only reach lane quadrant w % 4,
    // so warp w takes row (w % 4) * 32 + lane and half (w - 2) / 4 of the
    // stage's 8 words
    const int arow = (warp & 3) * 32 + lane, apart = (warp - 2) >> 2;
    const uint32_t alane = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const int n = n0 + arow;
    const bool nvalid = n < p.N;
    const uint32_t *qrow = reinterpret_cast<const uint32_t *>(p.qw) + static_cast<size_t>(n) * Kw;
    const int bm = dq & 63, bpair = dq >> 6;          // B: token, pair of 16-byte chunks
    // register ring of PD prefetched stages of 4 packed words; a word past
    // K or past N holds nibbles 8 (value 0)
    uint32_t ra[PD][4];
    auto fetch = [&](int kb, uint32_t (&w)[4]) {
#pragma unroll
      for (int i = 0; i < 4; ++i) w[i] = 0x88888888u;
      const int w0 = kb * 8 + apart * 4;
      if (!nvalid || kb >= kb1 || w0 >= Kw) return;
      if (!W4A16_IN_BOUNDS(n < p.N && w0 >= 0, p.status)) return;
      if (w0 + 4 <= Kw) {
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(qrow + w0));
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
      } else {
        for (int i = 0; i < 4 && w0 + i < Kw; ++i) w[i] = __ldg(qrow + w0 + i);
      }
    };
#pragma unroll
    for (int u = 0; u < PD; ++u) fetch(kb0 + u, ra[u]);
    int it = 0;
    bool ok = true;
    for (int kbase = kb0; kbase < kb1 && ok; kbase += PD) {
#pragma unroll
      for (int u = 0; u < PD; ++u) {
        const int kb = kbase + u;
        if (kb >= kb1) break;
        const int s = it % NS;
        const uint32_t ph = static_cast<uint32_t>(it / NS) & 1u;
        const int xs = it % FX_NSX;
        const uint32_t xph = static_cast<uint32_t>(it / FX_NSX) & 1u;
        ++it;
        uint32_t cw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) cw[i] = ra[u][i];
        fetch(kb + PD, ra[u]);
        // the slot is free, then the activation tile has landed
        int got = 1;
        if (lane == 0)
          got = mbar_wait(&empty[s], ph ^ 1u) && mbar_wait(&xfull[xs], xph) && !aborted(abort_flag);
        if (!__shfl_sync(0xFFFFFFFFu, got, 0)) { fail(); ok = false; break; }
        uint8_t *st = smem + s * SB;
        {
          tc_fence_after();  // the MMAs that read this A stage are complete
          uint32_t a[16];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint4 d = dequant_word_int(cw[i], magic, bias);
            a[4 * i] = d.x; a[4 * i + 1] = d.y; a[4 * i + 2] = d.z; a[4 * i + 3] = d.w;
          }
          tmem_st_16cols(alane + FX_A_COL0 + s * 32 + apart * 16, a);
        }
        // the fp32 tile: two [64 tokens][32 columns] halves, 16-byte pieces
        // of each 128-byte row swizzled by the row index
        const uint8_t *xt = xring + xs * FX_X_BYTES;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int chunk = bpair * 2 + j;
          const uint8_t *xrow = xt + (chunk >> 2) * (FX_X_BYTES / 2) + bm * 128;
          const int p0 = (chunk & 3) * 2;  // first 16-byte piece of the chunk
          const float4 lo = *reinterpret_cast<const float4 *>(xrow + ((p0 ^ (bm & 7)) << 4));
          const float4 hi = *reinterpret_cast<const float4 *>(xrow + (((p0 + 1) ^ (bm & 7)) << 4));
          const float v[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
          uint4 o1, o2, o3;
          split_chunk(v, o1, o2, o3);
          const uint32_t off = sw128_offset(bm, chunk);
          // the three 16-byte pieces inside the stage's three B tiles
          (void)W4A16_IN_BOUNDS(off + 16u <= static_cast<uint32_t>(FX_B_BYTES), p.status);
          *reinterpret_cast<uint4 *>(st + off) = o1;
          *reinterpret_cast<uint4 *>(st + FX_B_BYTES + off) = o2;
          *reinterpret_cast<uint4 *>(st + 2 * FX_B_BYTES + off) = o3;
        }
        tmem_store_wait();
        tc_fence_before();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&full[s]);
          mbar_arrive(&xempty[xs]);  // this warp has split its part of the tile
        }
      }
    }
  } else {
    // ------------------------------------------------------------ readback
    const int q = warp & 3;            // TMEM lane quadrant
    const int r = q * 32 + lane;       // weight row of the tile
    const int n = n0 + r;
    const bool nvalid = n < p.N;
    const float *srow = p.sc + static_cast<size_t>(nvalid ? n : 0) * G;
    float acc[FX_BM];
#pragma unroll
    for (int m = 0; m < FX_BM; ++m) acc[m] = 0.f;
    const int g_begin = 2 * kb0, g_end = min(G32, 2 * kb1);
    (void)W4A16_IN_BOUNDS(!nvalid || g_end == g_begin || ((g_end - 1) >> gsh) < G, p.status);
    float s_next = (nvalid && g_begin < g_end) ? __ldg(srow + (g_begin >> gsh)) : 0.f;
    bool ok = true;
    for (int gk = g_begin, g = 0; gk < g_end; ++gk, ++g) {
      const float s = s_next;  // the scale of 32-column group gk
      s_next = (nvalid && gk + 1 < g_end) ? __ldg(srow + ((gk + 1) >> gsh)) : 0.f;
      const int buf = g % FX_ACC;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&acc_full[buf], static_cast<uint32_t>(g / FX_ACC) & 1u))) {
        fail();
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + buf * FX_NB;
      // the group sum (all three pieces) times the group scale
#pragma unroll
      for (int part = 0; part < FX_BM / 16; ++part) {
        uint32_t d[16];
        tmem_ld_16cols(taddr + part * 16, d);
#pragma unroll
        for (int j = 0; j < 16; ++j)
          acc[part * 16 + j] = fmaf(s, __uint_as_float(d[j]), acc[part * 16 + j]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
    }
    if (ok) {
      // partial tile to shared memory (the pipeline stages are idle once
      // every group has been read): row r at red[r * FX_RED_LD], 16-byte
      // stores; the padded stride puts 8 consecutive rows' chunks in 8
      // different bank groups
      float *red = reinterpret_cast<float *>(smem) + r * FX_RED_LD;
#pragma unroll
      for (int m = 0; m < FX_BM; m += 4)
        *reinterpret_cast<float4 *>(red + m) = make_float4(acc[m], acc[m + 1], acc[m + 2], acc[m + 3]);
      fence_proxy_async_smem();  // the bulk copies below read the tile
    }
    __syncwarp();
  }

  __syncthreads();
  // ------------------------------------------------ split-K reduction (push)
  // every rank has parked its partial tile (a failed rank sends whatever
  // its tile holds: the status word already records the failure)
  cluster_wait();  // phase A: every rank's barriers are initialised
  const float *red = reinterpret_cast<const float *>(smem);
  if (threadIdx.x == 0 && ks > 1) push_send<FX_ROWS, FX_RED_LD>(red, recv, red_bar, rank, ks);
  griddep_wait();  // every thread may write y below
  if (ks > 1 && !mbar_wait(red_bar, 0)) fail();
  __syncwarp();
  cluster_arrive();  // phase B: the slices of this rank's rows have landed
  if (*reinterpret_cast<volatile int *>(abort_flag) == 0)
    push_owner_sum<FX_ROWS, FX_BM, FX_RED_LD, FX_MAX_KS>(red, recv, rank, ks, n0, 0, p.M, p.N, p.y,
                                                         p.ybf16, p.status);
  cluster_wait();  // phase B: every slice this CTA sent has landed
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(FX_TMEM_COLS)
                 : "memory");
  }
}

int env_int(const char *name) {
  const char *v = getenv(name);
  return v ? atoi(v) : 0;
}

}  // namespace

bool tc_f32_supported(int M, int N, int K) {
  return M > 0 && M <= FX_BM && N > 0 && K > 0 && K % 32 == 0;
}

cudaError_t launch_tc_f32(const float *x, const int32_t *qw, const float *sc, int M, int N, int K,
                          int group, void *y, bool y_bf16, bool overlap, cudaStream_t stream) {
  if (!tc_f32_supported(M, N, K)) return cudaErrorInvalidValue;
  const DeviceInfo &di = device_info();
  auto encode = encode_fn();
  if (encode == nullptr) return cudaErrorNotSupported;
  CUtensorMap tmap;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 4};
  const cuuint32_t box[2] = {FX_BK / 2, FX_BM};  // 128-byte rows
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(x), dims,
                      strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  FxParams p{};
  p.qw = qw;
  p.sc = sc;
  p.y = y;
  p.ybf16 = y_bf16 ? 1 : 0;
  p.M = M;
  p.N = N;
  p.K = K;
  p.num_tiles = (N + FX_ROWS - 1) / FX_ROWS;
  p.gs = group == 128 ? 7 : group == 64 ? 6 : 5;
  p.status = di.status;
  // split K over a cluster of up to 4 CTAs (a power of two: the split-K
  // slices are equal) so that the tiles cover the SMs once (the fp32 chain
  // of group sums is then at most 128 terms long for K <= 16384)
  static const int env_ks = env_int("W4A16_TC_KS");
  const int nk = (K + FX_BK - 1) / FX_BK;
  const int ks_cap = std::min(std::min(env_ks > 0 ? std::min(env_ks, FX_MAX_KS) : FX_MAX_KS, nk),
                              di.num_sms / std::max(1, p.num_tiles));
  int ks = 1;
  while (2 * ks <= ks_cap) ks *= 2;
  auto kern = tc_f32_kernel;
  static PerDeviceOnce attr_once;
  const cudaError_t attr_err = attr_once.run(
      [&] { return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, FX_SMEM); });
  if (attr_err != cudaSuccess) return attr_err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.num_tiles, ks);
  cfg.blockDim = dim3(FX_THREADS);
  cfg.dynamicSmemBytes = FX_SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = ks;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = overlap ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, tmap, p);
}

}  // namespace w4a16
