// Decode GEMV on CUDA cores (one token), built for back-to-back calls:
//   y[n] = sum_k x[k] * (nibble(n,k) - 8) * sc[n][k/g].
//
// One CTA per SM owns a contiguous block of weight rows. Its footprint (16
// warps, at most 64 registers a thread, a little under half of the shared
// memory) leaves room for the CTA of the NEXT call on the stream to sit
// beside it. Launched with programmatic stream serialisation, that next CTA
// starts as soon as it is resident: it requests its own weight rows into a
// ring of shared-memory stages and only then waits for the previous kernel
// to complete. The activations are read, and y written, after that wait. In
// a decode loop the weight stream of one call therefore runs under the
// unpack and FMA work of the call before it, and each call's critical path
// is the compute on rows that are already on chip.
//
// Work split. Warps own slices of K; a lane owns one or two packed words (8
// or 16 input columns, always inside one group) and keeps those activations
// in registers for the whole call. With K = 7168 (896 words) warps 0..11
// take two words per lane and warps 12..15 one, so each of the four warp
// schedulers of the SM (warp w runs on scheduler w mod 4) gets three
// two-word warps and one one-word warp: equal work per scheduler.
// There is no producer warp: thread 0 issues the first stages and, two
// stages ahead of its own warp, the refills of freed slots.
//
// Per stage (4 weight rows) a lane unpacks its words exactly into packed
// fp32 pairs (unpack8_pair: the same nibble of two words of one row for a
// two-word lane, of the same word of two rows for a one-word lane),
// multiplies with packed fp32 FMAs, scales each row's partial by its group
// scale and takes part in a fixed-order 4-row transpose reduction over the
// warp. The warps' row sums meet in a shared-memory table that the CTA adds
// in warp order at the end, so results are deterministic.
//
// Format: "The Quiet Commit: How a Single Documentation Edit Marks the
// Completion of a Major Engineering Milestone", section "The INT4 Milestone"
// (8 nibbles per int32 along K, value = nibble - 8, fp32 group scales).
// Accumulation in fp32: "The Silence of Success: A Single Line That Speaks
// Volumes", section "Assumptions Embedded in the Code".
#include <algorithm>
#include <cstdlib>
#include <mutex>
#include <type_traits>

#include "kernels.h"
#include "stream_core.cuh"

namespace w4a16 {

namespace {

constexpr int kGvWarps = 16;
constexpr int kGvThreads = 32 * kGvWarps;
constexpr int kGvRows = 4;            // weight rows per stage
constexpr int kGvMaxStages = 8;       // ring slots
constexpr int kGvMaxRowsPerCta = 64;  // bounds the table of per-warp row sums
// Shared memory one CTA may take so that two fit on an SM (228 KB per SM,
// 1 KB of it reserved per resident CTA).
constexpr size_t kGvSmemBudget = 110u * 1024u;

struct GemvParams {
  const void *x;
  const int32_t *qw;
  const float *sc;
  int N, K;
  void *y;     // fp32, or bf16 when ybf16
  int ybf16;
  int nstages; // ring slots
  int nwide;   // warps 0 .. nwide-1 take two words per lane, the others one
  int gs;      // log2 of the group size (5, 6 or 7)
  int srow;    // bytes per scale row, a multiple of 16
  int fault;   // testing aid: issue no weight copies (the waits then time out)
  int *status;
};

// Activations of one word (8 columns from k0), fp32 or bf16 -> fp32 x[8].
template <bool BF16>
__device__ __forceinline__ void load_x8(const void *x, int k0, bool active, float (&xv)[8]) {
  if (!active) {
#pragma unroll
    for (int j = 0; j < 8; ++j) xv[j] = 0.f;
    return;
  }
  if constexpr (BF16) {
    const uint4 u = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(x) + k0));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      xv[2 * h] = __uint_as_float(w[h] << 16);
      xv[2 * h + 1] = __uint_as_float(w[h] & 0xFFFF0000u);
    }
  } else {
    const float4 *src = reinterpret_cast<const float4 *>(static_cast<const float *>(x) + k0);
    const float4 p = __ldg(src), q = __ldg(src + 1);
    xv[0] = p.x; xv[1] = p.y; xv[2] = p.z; xv[3] = p.w;
    xv[4] = q.x; xv[5] = q.y; xv[6] = q.z; xv[7] = q.w;
  }
}

// Sum v[0..3] over the 32 lanes in a fixed order. On return a lane holds the
// full sum of row 2 * bit4(lane) + bit3(lane).
__device__ __forceinline__ float gv_reduce4(const float (&v)[4], int lane) {
  const bool b4 = lane & 16, b3 = lane & 8;
  const float q0 = (b4 ? v[2] : v[0]) + __shfl_xor_sync(0xFFFFFFFFu, b4 ? v[0] : v[2], 16);
  const float q1 = (b4 ? v[3] : v[1]) + __shfl_xor_sync(0xFFFFFFFFu, b4 ? v[1] : v[3], 16);
  float r = (b3 ? q1 : q0) + __shfl_xor_sync(0xFFFFFFFFu, b3 ? q0 : q1, 8);
  r += __shfl_xor_sync(0xFFFFFFFFu, r, 4);
  r += __shfl_xor_sync(0xFFFFFFFFu, r, 2);
  r += __shfl_xor_sync(0xFFFFFFFFu, r, 1);
  return r;
}

struct GvShared {
  uint64_t full[kGvMaxStages];   // stage landed (one arrival + transaction bytes)
  uint64_t empty[kGvMaxStages];  // every warp is done with the slot (one arrival per warp)
  int slot_stage[kGvMaxStages];  // last stage issued into the slot (-1: none)
  int abort;
};

template <bool BF16>
__global__ void __launch_bounds__(kGvThreads, 2) gemv_kernel(const GemvParams p) {
  constexpr int RS = kGvRows;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ GvShared sh;

  const int K = p.K;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t qrow = static_cast<uint32_t>(K) >> 1;  // bytes per packed row
  const uint32_t srow = static_cast<uint32_t>(p.srow);
  const uint32_t qstage = RS * qrow;
  const uint32_t stage_bytes = qstage + RS * srow;
  const int NS = p.nstages;

  const int r0 = static_cast<int>((static_cast<long long>(p.N) * blockIdx.x) / gridDim.x);
  const int r1 = static_cast<int>((static_cast<long long>(p.N) * (blockIdx.x + 1)) / gridDim.x);
  const int nrows = r1 - r0;
  const int nst = (nrows + RS - 1) / RS;

  uint8_t *stages = smem;
  float *red = reinterpret_cast<float *>(smem + NS * stage_bytes);  // [nst*RS][kGvWarps]

  // Request stage s into its slot (rows past the block are not copied; the
  // slot keeps stale bytes there whose sums are never stored).
  auto issue = [&](int s) {
    const int slot = s % NS;
    const int row = r0 + s * RS;
    const int rows = min(RS, r1 - row);
    uint8_t *dst = stages + slot * stage_bytes;
    const uint32_t bq = rows * qrow, bs = rows * srow;
    sh.slot_stage[slot] = s;
    // rows [row, row + rows) of qw and sc, into a stage of RS rows
    if (!W4A16_IN_BOUNDS(row >= 0 && rows > 0 && rows <= RS && row + rows <= p.N, p.status))
      return;  // the stage never fills: its waits time out
    mbar_arrive_expect_tx(&sh.full[slot], bq + bs);
    bulk_g2s(dst, reinterpret_cast<const uint8_t *>(p.qw) + static_cast<size_t>(row) * qrow, bq,
             &sh.full[slot]);
    bulk_g2s(dst + qstage,
             reinterpret_cast<const uint8_t *>(p.sc) + static_cast<size_t>(row) * srow, bs,
             &sh.full[slot]);
  };

  griddep_launch_dependents();
  if (threadIdx.x == 0) {
    sh.abort = 0;
    for (int i = 0; i < NS; ++i) {
      mbar_init(&sh.full[i], 1);
      mbar_init(&sh.empty[i], kGvWarps);
      sh.slot_stage[i] = -1;
    }
    fence_mbar_init();
    // The weights are not written by the previous kernel on the stream (the
    // overlap contract), so they are requested before waiting for it.
    if (!p.fault)
      for (int s = 0; s < min(NS, nst); ++s) issue(s);
  }
  __syncthreads();
  // x and y may be operands of the previous kernel: touch them only after it
  // has completed. Without programmatic launch this returns at once.
  griddep_wait();

  // This lane's words: two-word warps first, then one-word warps.
  const bool wide = warp < p.nwide;
  const int word0 = wide ? (warp * 64 + lane * 2) : (p.nwide * 64 + (warp - p.nwide) * 32 + lane);
  const int KW = K >> 3;
  const bool active = word0 < KW;  // KW % 4 == 0, so a two-word lane is all in or all out
  const int wc = active ? word0 : 0;  // inactive lanes read valid smem and weigh zero
  const int g = (wc << 3) >> p.gs;
  const PairUnpack uk = make_pair_unpack();

  // Refills: stage t >= NS goes into the slot of stage t - NS once every
  // warp has released that one. Thread 0 issues refill t when its own warp
  // is about to take stage t - NS + lead (a bounded wait on the slot's
  // `empty` barrier, short since the warps move through the stages
  // together), which leaves NS - lead stages of time for the copy to land.
  const int lead = max(1, min(2, NS - 1));  // stage t - NS must be behind warp 0
  auto wait_stage = [&](int s) -> bool {
    if (threadIdx.x == 0 && !p.fault) {
      const int t = s + NS - lead;
      if (t >= NS && t < nst) {
        if (!mbar_wait_or_abort(&sh.empty[(t - NS) % NS], static_cast<uint32_t>((t - NS) / NS) & 1u,
                                &sh.abort)) {
          if (atomicExch(&sh.abort, 1) == 0) record_status(p.status, W4A16_ERR_TIMEOUT);
        } else {
          fence_proxy_async_smem();
          issue(t);
        }
      }
    }
    // every lane waits for the stage itself (one shared word, broadcast); a
    // stage that has landed costs one non-blocking test
    const uint32_t par = static_cast<uint32_t>(s / NS) & 1u;
    if (mbar_test_wait(&sh.full[s % NS], par) ||
        mbar_wait_or_abort(&sh.full[s % NS], par, &sh.abort))
      return true;
    if (lane == 0 && atomicExch(&sh.abort, 1) == 0) record_status(p.status, W4A16_ERR_TIMEOUT);
    return false;
  };
  // Release a slot that a later stage refills (the arrive orders the warp's
  // reads of it before the refill).
  auto release = [&](int s) {
    if (s + NS < nst) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.empty[s % NS]);
    }
  };
  auto store_rows = [&](int s, const float (&part)[RS]) {
    const float res = gv_reduce4(part, lane);
    if ((lane & 7) == 0) {
      const int row = s * RS + (lane >> 3);
      if (row < nrows) red[row * kGvWarps + warp] = res;
    }
  };

  if (wide) {
    // Two consecutive words per lane (16 columns): the pair holds the same
    // nibble of both words; x pair j = (column j of word 0, of word 1).
    uint64_t xp[8];
    {
      float x0[8], x1[8];
      const bool xin = W4A16_IN_BOUNDS(!active || wc * 8 + 16 <= p.K, p.status);
      load_x8<BF16>(p.x, wc * 8, active && xin, x0);
      load_x8<BF16>(p.x, wc * 8 + 8, active && xin, x1);
#pragma unroll
      for (int j = 0; j < 8; ++j) xp[j] = pack_f32x2(x0[j], x1[j]);
    }
    for (int s = 0; s < nst; ++s) {
      if (!wait_stage(s)) break;
      const uint8_t *st = stages + (s % NS) * stage_bytes;
      // all of the stage's words and scales first, then the arithmetic
      uint2 w[RS];
      float sv[RS];
#pragma unroll
      for (int r = 0; r < RS; ++r) {
        w[r] = *reinterpret_cast<const uint2 *>(st + r * qrow + wc * 4);
        sv[r] = reinterpret_cast<const float *>(st + qstage + r * srow)[g];
      }
      float part[RS];
#pragma unroll
      for (int r = 0; r < RS; ++r) {
        uint64_t v[8];
        unpack8_pair(w[r].x, w[r].y, uk, v);
        uint64_t acc = 0ull;
#pragma unroll
        for (int j = 0; j < 8; ++j) acc = fma_f32x2(v[j], xp[j], acc);
        float lo, hi;
        unpack_f32x2(acc, lo, hi);
        part[r] = (lo + hi) * sv[r];
      }
      release(s);
      store_rows(s, part);
    }
  } else {
    // One word per lane (8 columns): the pair holds the same nibble of two
    // rows; x pair j = (column j, column j).
    uint64_t xd[8];
    {
      float x0[8];
      const bool xin = W4A16_IN_BOUNDS(!active || wc * 8 + 8 <= p.K, p.status);
      load_x8<BF16>(p.x, wc * 8, active && xin, x0);
#pragma unroll
      for (int j = 0; j < 8; ++j) xd[j] = pack_f32x2(x0[j], x0[j]);
    }
    for (int s = 0; s < nst; ++s) {
      if (!wait_stage(s)) break;
      const uint8_t *st = stages + (s % NS) * stage_bytes;
      uint32_t w[RS];
      float sv[RS];
#pragma unroll
      for (int r = 0; r < RS; ++r) {
        w[r] = *reinterpret_cast<const uint32_t *>(st + r * qrow + wc * 4);
        sv[r] = reinterpret_cast<const float *>(st + qstage + r * srow)[g];
      }
      float part[RS];
#pragma unroll
      for (int r = 0; r < RS; r += 2) {
        const float sa = sv[r], sb = sv[r + 1];
        uint64_t v[8];
        unpack8_pair(w[r], w[r + 1], uk, v);
        uint64_t acc = 0ull;
#pragma unroll
        for (int j = 0; j < 8; ++j) acc = fma_f32x2(v[j], xd[j], acc);
        float lo, hi;
        unpack_f32x2(acc, lo, hi);
        part[r] = lo * sa;
        part[r + 1] = hi * sb;
      }
      release(s);
      store_rows(s, part);
    }
  }

  __syncthreads();
  if (static_cast<volatile int &>(sh.abort) != 0) {
    // Let copies still in flight land before the CTA exits (bounded waits;
    // a landed copy completes at once).
    if (threadIdx.x == 0)
      for (int i = 0; i < NS; ++i)
        if (sh.slot_stage[i] >= 0)
          mbar_wait(&sh.full[i], static_cast<uint32_t>(sh.slot_stage[i] / NS) & 1u);
    return;
  }
  if (threadIdx.x < nrows) {
    const float *v = red + threadIdx.x * kGvWarps;
    float a = 0.f;
#pragma unroll
    for (int w = 0; w < kGvWarps; ++w) a += v[w];
    if (W4A16_IN_BOUNDS(r0 + static_cast<int>(threadIdx.x) < p.N, p.status))
      store_y(p.y, static_cast<size_t>(r0 + threadIdx.x), a, p.ybf16);
  }
}

int gv_env(const char *name) {
  const char *v = getenv(name);
  return v ? atoi(v) : 0;
}

template <bool BF16>
cudaError_t gemv_set_smem(int bytes) {
  static PerDeviceOnce once;
  return once.run([&] {
    cudaError_t e = cudaFuncSetAttribute(gemv_kernel<BF16>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gemv_kernel<BF16>, cudaFuncAttributePreferredSharedMemoryCarveout,
                               100);
    return e;
  });
}

}  // namespace

bool gemv_supported(int M, int N, int K, int group) {
  if (M != 1 || N <= 0 || K <= 0 || K % 32 != 0 || K > kGemvMaxK) return false;
  if (K % group != 0) return false;
  return (K / group) % 4 == 0;  // scale rows of whole 16-byte units
}

cudaError_t launch_gemv(const void *x, bool x_bf16, const int32_t *qw, const float *sc, int N,
                        int K, int group, void *y, bool y_bf16, bool overlap,
                        cudaStream_t stream) {
  const DeviceInfo &di = device_info();
  GemvParams p{};
  p.x = x;
  p.qw = qw;
  p.sc = sc;
  p.N = N;
  p.K = K;
  p.y = y;
  p.ybf16 = y_bf16 ? 1 : 0;
  p.gs = group == 128 ? 7 : group == 64 ? 6 : 5;
  p.srow = (K >> p.gs) * 4;
  p.status = di.status;
  p.fault = take_injected_fault() ? 1 : 0;
  // 32-word columns of K: up to 16 warps of one word per lane, beyond that
  // the first (units - 16) warps take two.
  const int units = (K / 8 + 31) / 32;
  p.nwide = units > kGvWarps ? units - kGvWarps : 0;

  static const int env_ctas = gv_env("W4A16_GEMV_CTAS");
  int G = std::min((N + kGvRows - 1) / kGvRows, env_ctas > 0 ? env_ctas : di.num_sms);
  G = std::max({1, G, (N + kGvMaxRowsPerCta - 1) / kGvMaxRowsPerCta});
  const int rows = (N + G - 1) / G;
  const int nst = (rows + kGvRows - 1) / kGvRows;
  const size_t stage = static_cast<size_t>(kGvRows) * (K / 2 + p.srow);
  const size_t table = static_cast<size_t>(nst) * kGvRows * kGvWarps * sizeof(float);
  static const int env_ns = gv_env("W4A16_GEMV_NS");
  int ns = std::min({nst, kGvMaxStages, env_ns > 0 ? env_ns : kGvMaxStages});
  while (ns > 1 && ns * stage + table > kGvSmemBudget) --ns;
  const size_t smem = ns * stage + table;
  if (smem > static_cast<size_t>(di.smem_optin) - 1024) return cudaErrorInvalidConfiguration;
  p.nstages = ns;

  cudaError_t e = x_bf16 ? gemv_set_smem<true>(static_cast<int>(kGvSmemBudget))
                         : gemv_set_smem<false>(static_cast<int>(kGvSmemBudget));
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = overlap ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(G);
  cfg.blockDim = dim3(kGvThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return x_bf16 ? cudaLaunchKernelEx(&cfg, gemv_kernel<true>, p)
                : cudaLaunchKernelEx(&cfg, gemv_kernel<false>, p);
}

}  // namespace w4a16
