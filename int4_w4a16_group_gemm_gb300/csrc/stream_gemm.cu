// Small-M W4A16 GEMM on CUDA cores: the memory-bound decode / tree-verify
// kernel. y[m][n] = sum_k x[m][k] * (nibble(n,k) - 8) * sc[n][k/32].
//
// The grid is row blocks x token tiles. A CTA owns a contiguous range of
// weight rows and up to 3 tokens. Because qw and sc are row-major, the row
// range is one contiguous run of bytes in each tensor, so a producer warp
// streams it into a ring of shared-memory stages with 1-D bulk copies (8
// rows per stage, the whole ring in flight from the first cycle), and the
// consumer warps unpack and multiply (see stream_core.cuh for the split of
// K over warps and lanes). The per-warp row sums are combined across the
// CTA's warps in a fixed order, so results are deterministic. Token tiles
// of the same rows re-read the weights, from L2 when they fit there.
//
// Format: "The Quiet Commit: How a Single Documentation Edit Marks the
// Completion of a Major Engineering Milestone", section "The INT4 Milestone"
// (8 nibbles per int32 along K, value = nibble - 8, fp32 group scales).
// Accumulation in fp32: "The Silence of Success: A Single Line That Speaks
// Volumes", section "Assumptions Embedded in the Code".
#include <algorithm>
#include <cstdlib>
#include <mutex>

#include "kernels.h"
#include "stream_core.cuh"

namespace w4a16 {

namespace {

struct StreamParams {
  const void *x;
  int ldx;
  int M;  // tokens; CTA row blockIdx.y covers tokens [MT*blockIdx.y, MT*blockIdx.y + MT)
  const int32_t *qw;
  const float *sc;
  int N, K;
  void *y;      // fp32, or bf16 when ybf16
  int ybf16;
  int ldy;
  int nstages;
  int gs;       // log2 of the group size (5, 6 or 7)
  int srow;     // bytes per scale row: (K / group) * 4
  int sc_bulk;  // 1: scales staged by bulk copy (scale rows a multiple of 16 bytes)
  int fault;    // testing aid: skip the weight copies (waits then time out)
  int prewait;  // stages of the first ring fill requested before the programmatic wait
  int *status;
};

// Largest row block of a CTA (bounds the table of per-warp row sums).
constexpr int kMaxRowsPerCta = 128;

// Roles: warps 0 .. nw-1 consume (each owns one K-slice of every row, see
// stream_core.cuh) and the last warp produces: it issues the bulk copies
// into the ring of stages and refills a stage as soon as every consumer has
// loaded its words from it (the stage's `empty` mbarrier). Consumers never
// wait for each other. Up to two tokens, each keeps one chunk in flight:
// the cross-lane reduction of chunk c is issued together with the FMAs of
// chunk c + 1. The per-warp row sums go to a shared-memory table that holds
// every row of the CTA. After the last chunk the whole CTA adds the table
// over the warps in a fixed order and writes y.
template <int MT, int WPL, bool BF16, bool SCB, int MAXW, int MINB>
__global__ void __launch_bounds__(32 * MAXW, MINB) stream_gemm_kernel(const StreamParams p) {
  constexpr int EPL = 8 * WPL;
  constexpr int SLICE = 32 * EPL;
  constexpr int RC = kRowsPerChunk;
  constexpr bool kDeferReduce = MT <= 2;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_abort;

  const int K = p.K;
  const int nw = (blockDim.x >> 5) - 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t qrow = static_cast<uint32_t>(K) >> 1;  // bytes per packed row
  const uint32_t srow = static_cast<uint32_t>(p.srow);  // bytes per scale row
  const uint32_t qstage = RC * qrow;
  const uint32_t stage_bytes = qstage + (SCB ? RC * srow : 0u);
  const int NS = p.nstages;
  const int m0 = blockIdx.y * MT;
  const int mt = min(MT, p.M - m0);

  const int r0 = static_cast<int>((static_cast<long long>(p.N) * blockIdx.x) / gridDim.x);
  const int r1 = static_cast<int>((static_cast<long long>(p.N) * (blockIdx.x + 1)) / gridDim.x);
  const int nchunks = (r1 - r0 + RC - 1) / RC;

  // shared memory: NS stages | full[NS] | empty[NS] | red[nchunks*RC][MT][nw]
  uint8_t *stages = smem;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + NS * stage_bytes);
  uint64_t *empty = full + NS;
  float *red = reinterpret_cast<float *>(empty + NS);

  auto issue = [&](int c) {
    const int slot = c % NS;
    const int row = r0 + c * RC;
    const int rows = min(RC, r1 - row);
    uint8_t *dst = stages + slot * stage_bytes;
    const uint32_t bq = rows * qrow;
    const uint32_t bs = SCB ? rows * srow : 0u;
    // rows [row, row + rows) of qw and sc, into a stage of RC rows
    if (!W4A16_IN_BOUNDS(row >= 0 && rows > 0 && rows <= RC && row + rows <= p.N, p.status))
      return;  // the stage never fills: its waits time out
    mbar_arrive_expect_tx(&full[slot], bq + bs);
    bulk_g2s(dst, reinterpret_cast<const uint8_t *>(p.qw) + static_cast<size_t>(row) * qrow, bq,
             &full[slot]);
    if (SCB)
      bulk_g2s(dst + qstage, reinterpret_cast<const uint8_t *>(p.sc) + static_cast<size_t>(row) * srow,
               bs, &full[slot]);
  };

  // The producer's lane 0 sets up the ring and starts the weight stream at
  // once: the weights are not written by the previous kernel on the stream
  // (the overlap contract), so they may be read before it has finished. It
  // requests `prewait` stages now and the rest of the first fill after the
  // wait.
  const int ninit = p.fault ? 0 : min(NS, nchunks);  // the first ring fill
  const int first = min(ninit, p.prewait);            // requested before the wait
  if (threadIdx.x == nw * 32) {
    s_abort = 0;
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], nw);
    }
    fence_mbar_init();
    for (int c = 0; c < first; ++c) issue(c);
  }
  __syncthreads();
  // Let the next kernel start launching, then wait for the previous one
  // before touching x or y (both may be its operands). Without programmatic
  // launch both calls are no-ops.
  griddep_launch_dependents();
  griddep_wait();

  if (warp == nw) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      for (int c = first; c < ninit; ++c) issue(c);
      int issued = ninit, released = 0;
      for (int c = 0; c + NS < nchunks && !p.fault; ++c) {
        if (!mbar_wait_or_abort(&empty[c % NS], static_cast<uint32_t>(c / NS) & 1u, &s_abort)) {
          if (atomicExch(&s_abort, 1) == 0) record_status(p.status, W4A16_ERR_TIMEOUT);
          break;
        }
        released = c + 1;
        issue(c + NS);
        ++issued;
      }
      // After an abort, let the copies still in flight land before the CTA
      // exits (each wait is bounded; a landed copy completes at once).
      if (static_cast<volatile int &>(s_abort) != 0)
        for (int d = released; d < issued; ++d)
          mbar_wait(&full[d % NS], static_cast<uint32_t>(d / NS) & 1u);
    }
  } else {
    // ------------------------------------------------------------ consumers
    const NibbleConsts nk = make_nibble_consts();
    // This lane's columns and its activations (kept in registers).
    const int k0 = warp * SLICE + lane * EPL;
    const bool active = k0 < K;
    const int kc = active ? k0 : 0;  // inactive lanes read valid smem, weigh zero
    const int g = kc >> p.gs;  // a lane's columns lie in one group
    // this lane's words and scale inside every stage row
    (void)W4A16_IN_BOUNDS((kc >> 1) + 4 * WPL <= static_cast<int>(qrow) &&
                              (!SCB || g * 4 < static_cast<int>(srow)),
                          p.status);
    uint64_t xr[MT][EPL / 2];
#pragma unroll
    for (int t = 0; t < MT; ++t) {
      const void *xrow = nullptr;
      if (active && t < mt &&
          W4A16_IN_BOUNDS(m0 + t < p.M && k0 + EPL <= p.K && p.ldx >= p.K, p.status)) {
        const size_t off = static_cast<size_t>(m0 + t) * p.ldx;
        xrow = BF16 ? static_cast<const void *>(static_cast<const uint16_t *>(p.x) + off)
                    : static_cast<const void *>(static_cast<const float *>(p.x) + off);
      }
      load_x_slice<EPL, BF16>(xrow, k0, xr[t]);
    }

    // Wait for chunk c, copy this lane's words and scales of its 8 rows to
    // registers and release the stage. Rows past the CTA's range hold stale
    // bytes whose sums are never stored (the reduction keeps rows apart).
    auto fetch = [&](int c, uint32_t (&wd)[RC][WPL], float (&sv)[RC]) -> bool {
      const int slot = c % NS;
      const int row0 = r0 + c * RC;
      if (!SCB) {
        const int rows = min(RC, r1 - row0);
#pragma unroll
        for (int r = 0; r < RC; ++r)
          sv[r] = r < rows && W4A16_IN_BOUNDS(row0 + r < p.N && g < (K >> p.gs), p.status)
                      ? __ldg(reinterpret_cast<const float *>(
                                  reinterpret_cast<const uint8_t *>(p.sc) +
                                  static_cast<size_t>(row0 + r) * srow) + g)
                      : 0.f;
      }
      int ok = 1;
      if (lane == 0) {
        ok = mbar_wait_or_abort(&full[slot], static_cast<uint32_t>(c / NS) & 1u, &s_abort);
        if (!ok && atomicExch(&s_abort, 1) == 0) record_status(p.status, W4A16_ERR_TIMEOUT);
      }
      if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) return false;
      const uint8_t *st = stages + slot * stage_bytes;
      const uint8_t *wbase = st + (kc >> 1);
#pragma unroll
      for (int r = 0; r < RC; ++r) {
        load_words<WPL>(wbase + r * qrow, wd[r]);
        if (SCB) sv[r] = reinterpret_cast<const float *>(st + qstage + r * srow)[g];
      }
      // the loads above have returned once their values are used; order
      // them before the release with a warp barrier
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
      return true;
    };
    auto store_sums = [&](int c, const float (&part)[RC][MT]) {
      float res[MT];
      warp_reduce_8rows<MT>(part, res, lane);
      if ((lane & 3) == 0) {
        const int row = c * RC + ((lane >> 2) & 7);
#pragma unroll
        for (int t = 0; t < MT; ++t) red[(row * MT + t) * nw + warp] = res[t];
      }
    };

    uint32_t wd[RC][WPL];
    float sv[RC];
    if constexpr (kDeferReduce) {
      float prev[RC][MT];
      bool ok = nchunks > 0 && fetch(0, wd, sv);
      if (ok) rows_dot<MT, WPL>(wd, sv, xr, prev, nk);
      for (int c = 1; ok && c < nchunks; ++c) {
        ok = fetch(c, wd, sv);
        if (!ok) break;
        float part[RC][MT];
        rows_dot<MT, WPL>(wd, sv, xr, part, nk);
        store_sums(c - 1, prev);
#pragma unroll
        for (int r = 0; r < RC; ++r)
#pragma unroll
          for (int t = 0; t < MT; ++t) prev[r][t] = part[r][t];
      }
      if (ok && nchunks > 0) store_sums(nchunks - 1, prev);
    } else {
      // three tokens: no registers to spare for a chunk in flight
      for (int c = 0; c < nchunks; ++c) {
        if (!fetch(c, wd, sv)) break;
        float part[RC][MT];
        rows_dot<MT, WPL>(wd, sv, xr, part, nk);
        store_sums(c, part);
      }
    }
  }

  // ------------------------------------------------------------ epilogue
  // Every consumer's sums are in the table: add them over the warps in a
  // fixed order (warp 0 first) and write y.
  __syncthreads();
  if (static_cast<volatile int &>(s_abort) != 0) return;
  const int nrows = r1 - r0;
  for (int i = threadIdx.x; i < nrows * MT; i += blockDim.x) {
    const int row = i / MT, t = i - row * MT;
    if (t >= mt) continue;
    const float *v = red + static_cast<size_t>(i) * nw;
    float a = 0.f;
    for (int w = 0; w < nw; ++w) a += v[w];
    if (W4A16_IN_BOUNDS(m0 + t < p.M && r0 + row < p.N && p.ldy >= p.N, p.status))
      store_y(p.y, static_cast<size_t>(m0 + t) * p.ldy + r0 + row, a, p.ybf16);
  }
}

// Tuning overrides (read once): W4A16_STREAM_NS (stages, 1..8),
// W4A16_STREAM_CTAS (row blocks per SM, 1..4), W4A16_STREAM_PREWAIT (stages
// requested before the programmatic wait, 1..8); 0 = automatic.
int env_int(const char *name) {
  const char *v = getenv(name);
  return v ? atoi(v) : 0;
}

template <int MT, int WPL, bool BF16, bool SCB, int MAXW, int MINB>
cudaError_t launch_tiles(const StreamParams &base, int tiles, int N, int K, int nsm,
                         int smem_optin, bool overlap, cudaStream_t stream) {
  constexpr int SLICE = 32 * 8 * WPL;
  const int nw = (K + SLICE - 1) / SLICE;
  const int threads = (nw + 1) * 32;
  if (nw + 1 > MAXW) return cudaErrorInvalidConfiguration;
  StreamParams p = base;
  const size_t stage = kRowsPerChunk * (K / 2 + (SCB ? (K >> base.gs) * 4 : 0));
  static const int env_ns = env_int("W4A16_STREAM_NS");
  static const int env_ctas = env_int("W4A16_STREAM_CTAS");
  static const int env_prewait = env_int("W4A16_STREAM_PREWAIT");
  // MINB row blocks per SM (more when a block would exceed kMaxRowsPerCta
  // rows). The unpack is bound by instruction issue: two CTAs of 14
  // consumer warps keep all four schedulers of an SM equally busy, which
  // beats one CTA with the next call's CTA resident beside it.
  const int ctas_per_sm = env_ctas > 0 ? std::min(env_ctas, 4) : MINB;
  int gx = std::min((N + kRowsPerChunk - 1) / kRowsPerChunk, nsm * ctas_per_sm);
  gx = std::max({1, gx, (N + kMaxRowsPerCta - 1) / kMaxRowsPerCta});
  const int rows_per_cta = (N + gx - 1) / gx;
  const int want = std::max(1, (rows_per_cta + kRowsPerChunk - 1) / kRowsPerChunk);
  auto bytes_for = [&](int ns) {
    return static_cast<size_t>(ns) * stage + 2ull * ns * sizeof(uint64_t) +
           static_cast<size_t>(want) * kRowsPerChunk * MT * nw * sizeof(float);
  };
  const size_t budget = std::min<size_t>(static_cast<size_t>(smem_optin) - 1024,
                                         MINB >= 2 ? (227u * 1024u) / 2 - 2048 : 227u * 1024u);
  int ns = env_ns > 0 ? std::min(env_ns, 8) : std::min(want, 4);
  while (ns > 1 && bytes_for(ns) > budget) --ns;
  if (bytes_for(ns) > static_cast<size_t>(smem_optin) - 1024) return cudaErrorInvalidConfiguration;
  p.nstages = ns;
  // Only the first stage is requested before the programmatic wait: the
  // activation loads that follow the wait then queue behind one stage of
  // weights instead of the whole ring (decode GEMV: 7.4-7.5 against 7.8 us
  // per chained call with the whole ring requested first).
  p.prewait = env_prewait > 0 ? env_prewait : 1;
  const size_t smem = bytes_for(ns);
  auto kern = stream_gemm_kernel<MT, WPL, BF16, SCB, MAXW, MINB>;
  static PerDeviceOnce attr_once;
  const cudaError_t attr_err = attr_once.run([&] {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                smem_optin - 1024);
  });
  if (attr_err != cudaSuccess) return attr_err;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = overlap ? 1 : 0;
  for (int t0 = 0; t0 < tiles; t0 += 65535) {
    const int nt = std::min(tiles - t0, 65535);
    StreamParams q = p;
    q.M = std::min(p.M - t0 * MT, nt * MT);
    q.x = BF16 ? static_cast<const void *>(static_cast<const uint16_t *>(p.x) +
                                           static_cast<size_t>(t0) * MT * p.ldx)
               : static_cast<const void *>(static_cast<const float *>(p.x) +
                                           static_cast<size_t>(t0) * MT * p.ldx);
    q.y = static_cast<uint8_t *>(p.y) +
          static_cast<size_t>(t0) * MT * p.ldy * (p.ybf16 ? 2 : 4);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(gx, nt);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, q);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <int MT, int WPL, bool BF16, int MAXW, int MINB>
cudaError_t launch_tiles_sc(const StreamParams &p, int tiles, int N, int K, int nsm,
                            int smem_optin, bool overlap, cudaStream_t stream) {
  return p.sc_bulk
             ? launch_tiles<MT, WPL, BF16, true, MAXW, MINB>(p, tiles, N, K, nsm, smem_optin,
                                                             overlap, stream)
             : launch_tiles<MT, WPL, BF16, false, MAXW, MINB>(p, tiles, N, K, nsm, smem_optin,
                                                              overlap, stream);
}

}  // namespace

int max_k_stream(int mt) { return mt == 1 ? 16384 : 8192; }

// Largest K for token tiles of 2 or 3 (15 consumer warps of two packed
// words per lane, plus the producer: 16 warps keep 128 registers a thread).
constexpr int kMaxKMultiToken = 15 * 512;

int stream_tile(int M, int K) {
  // up to 3 tokens per CTA (two packed words per lane); one token per CTA
  // beyond kMaxKMultiToken (four words per lane up to K = 16384)
  return K > kMaxKMultiToken ? 1 : std::min(M, 3);
}

int stream_gemm_passes(int M, int K) {
  const int tiles = (M + stream_tile(M, K) - 1) / stream_tile(M, K);
  return (tiles + 65534) / 65535;
}

cudaError_t launch_stream_gemm(const void *x, bool x_bf16, int ldx, const int32_t *qw,
                               const float *sc, int M, int N, int K, int group, void *y, bool y_bf16, int ldy,
                               bool overlap, cudaStream_t stream) {
  const DeviceInfo &di = device_info();
  StreamParams p{};
  p.x = x;
  p.ldx = ldx;
  p.M = M;
  p.qw = qw;
  p.sc = sc;
  p.N = N;
  p.K = K;
  p.y = y;
  p.ybf16 = y_bf16 ? 1 : 0;
  p.ldy = ldy;
  p.gs = group == 128 ? 7 : group == 64 ? 6 : 5;
  p.srow = (K >> p.gs) * 4;
  p.sc_bulk = ((K >> p.gs) % 4 == 0) ? 1 : 0;
  p.status = di.status;
  p.fault = take_injected_fault() ? 1 : 0;
  const int mt = stream_tile(M, K);
  const int tiles = (M + mt - 1) / mt;
  const int nsm = di.num_sms, opt = di.smem_optin;
  // One token: lanes own two packed words per row (16 columns) up to
  // K = 7680, four beyond. Up to K = 7168 two CTAs (14 consumer warps and
  // the producer each, at most 64 registers a thread) share an SM.
  if (mt == 1 && K <= 7168)
    return x_bf16 ? launch_tiles_sc<1, 2, true, 15, 2>(p, tiles, N, K, nsm, opt, overlap, stream)
                  : launch_tiles_sc<1, 2, false, 15, 2>(p, tiles, N, K, nsm, opt, overlap, stream);
  if (mt == 1 && K <= kMaxKMultiToken)
    return x_bf16 ? launch_tiles_sc<1, 2, true, 16, 1>(p, tiles, N, K, nsm, opt, overlap, stream)
                  : launch_tiles_sc<1, 2, false, 16, 1>(p, tiles, N, K, nsm, opt, overlap, stream);
  if (mt == 1)
    return x_bf16 ? launch_tiles_sc<1, 4, true, 17, 1>(p, tiles, N, K, nsm, opt, overlap, stream)
                  : launch_tiles_sc<1, 4, false, 17, 1>(p, tiles, N, K, nsm, opt, overlap, stream);
  if (mt == 2)
    return x_bf16 ? launch_tiles_sc<2, 2, true, 16, 1>(p, tiles, N, K, nsm, opt, overlap, stream)
                  : launch_tiles_sc<2, 2, false, 16, 1>(p, tiles, N, K, nsm, opt, overlap, stream);
  return x_bf16 ? launch_tiles_sc<3, 2, true, 16, 1>(p, tiles, N, K, nsm, opt, overlap, stream)
                : launch_tiles_sc<3, 2, false, 16, 1>(p, tiles, N, K, nsm, opt, overlap, stream);
}

}  // namespace w4a16
