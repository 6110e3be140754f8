// Small-M W4A16 GEMM on CUDA cores: the memory-bound decode / tree-verify
// kernel. y[m][n] = sum_k x[m][k] * (nibble(n,k) - 8) * sc[n][k/32].
//
// Each CTA owns a contiguous range of weight rows. Because qw and sc are
// row-major, that range is one contiguous run of bytes in each tensor, so a
// single thread streams it into a ring of shared-memory stages with 1-D bulk
// copies (8 rows per stage, several stages in flight from the first cycle),
// and every warp consumes the stages (see stream_core.cuh for the split of
// K over warps and lanes). The per-warp row sums are combined across the
// CTA's warps in a fixed order, so results are deterministic.
//
// Format: "The Quiet Commit: How a Single Documentation Edit Marks the
// Completion of a Major Engineering Milestone", section "The INT4 Milestone"
// (8 nibbles per int32 along K, value = nibble - 8, fp32 group scales).
// Accumulation in fp32: "The Silence of Success: A Single Line That Speaks
// Volumes", section "Assumptions Embedded in the Code".
#include <algorithm>

#include "kernels.h"
#include "stream_core.cuh"

namespace w4a16 {

namespace {

struct StreamParams {
  const void *x;
  int ldx;
  int mt;  // valid tokens in this pass (<= MT)
  const int32_t *qw;
  const float *sc;
  int N, K;
  float *y;
  int ldy;
  int nstages;
  int sc_bulk;  // 1: scales staged by bulk copy (K % 128 == 0)
  int fault;    // testing aid: skip the weight copies (waits then time out)
  int *status;
};

template <int MT, int WPL, bool BF16>
__global__ void __launch_bounds__(stream_max_threads(MT), 1)
    stream_gemm_kernel(const StreamParams p) {
  constexpr int EPL = 8 * WPL;
  constexpr int SLICE = 32 * EPL;
  constexpr int RC = kRowsPerChunk;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_abort;

  const int K = p.K;
  const int nw = blockDim.x >> 5;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = K >> 5;
  const uint32_t qrow = static_cast<uint32_t>(K) >> 1;  // bytes per packed row
  const uint32_t srow = static_cast<uint32_t>(K) >> 3;  // bytes per scale row
  const uint32_t qstage = RC * qrow;
  const uint32_t stage_bytes = qstage + (p.sc_bulk ? RC * srow : 0u);
  const int NS = p.nstages;

  uint8_t *stages = smem;
  float *red = reinterpret_cast<float *>(smem + NS * stage_bytes);
  uint64_t *full = reinterpret_cast<uint64_t *>(red + 2 * nw * RC * MT);

  const int r0 = static_cast<int>((static_cast<long long>(p.N) * blockIdx.x) / gridDim.x);
  const int r1 = static_cast<int>((static_cast<long long>(p.N) * (blockIdx.x + 1)) / gridDim.x);
  const int nchunks = (r1 - r0 + RC - 1) / RC;

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < NS; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
  }
  __syncthreads();

  int issued = 0;  // meaningful in thread 0 only
  auto issue = [&](int c) {
    const int slot = c % NS;
    const int row = r0 + c * RC;
    const int rows = min(RC, r1 - row);
    uint8_t *dst = stages + slot * stage_bytes;
    const uint32_t bq = rows * qrow;
    const uint32_t bs = p.sc_bulk ? rows * srow : 0u;
    mbar_arrive_expect_tx(&full[slot], bq + bs);
    bulk_g2s(dst, reinterpret_cast<const uint8_t *>(p.qw) + static_cast<size_t>(row) * qrow, bq,
             &full[slot]);
    if (p.sc_bulk)
      bulk_g2s(dst + qstage, reinterpret_cast<const uint8_t *>(p.sc) + static_cast<size_t>(row) * srow,
               bs, &full[slot]);
  };
  if (threadIdx.x == 0 && !p.fault) {
    for (; issued < min(NS, nchunks); ++issued) issue(issued);
  }
  // The weights are in flight. Let the next kernel start launching, then
  // wait for the previous one before touching x or y (both may be its
  // operands). Without programmatic launch both calls are no-ops.
  griddep_launch_dependents();
  griddep_wait();

  // This lane's columns and its activations (kept in registers).
  const int k0 = warp * SLICE + lane * EPL;
  const bool active = k0 < K;
  const int g = k0 >> 5;
  float xr[MT][EPL];
#pragma unroll
  for (int t = 0; t < MT; ++t) {
    const void *xrow = nullptr;
    if (active && t < p.mt) {
      xrow = BF16 ? static_cast<const void *>(static_cast<const uint16_t *>(p.x) +
                                              static_cast<size_t>(t) * p.ldx)
                  : static_cast<const void *>(static_cast<const float *>(p.x) +
                                              static_cast<size_t>(t) * p.ldx);
    }
    load_x_slice<EPL, BF16>(xrow, k0, xr[t]);
  }

  int c = 0;
  for (; c < nchunks; ++c) {
    const int slot = c % NS;
    const uint32_t parity = static_cast<uint32_t>(c / NS) & 1u;
    const int row0 = r0 + c * RC;
    const int rows = min(RC, r1 - row0);
    bool ok = mbar_wait(&full[slot], parity);
    if (!ok) {
      record_status(p.status, W4A16_ERR_TIMEOUT);
      s_abort = 1;
    }
    const uint8_t *st = stages + slot * stage_bytes;

    float part[RC][MT];
#pragma unroll
    for (int r = 0; r < RC; ++r) {
      float acc[MT];
      if (ok && active && r < rows) {
        uint32_t wd[WPL];
        load_words<WPL>(st + r * qrow + (k0 >> 1), wd);
        const float s = p.sc_bulk
                            ? reinterpret_cast<const float *>(st + qstage + r * srow)[g]
                            : __ldg(p.sc + static_cast<size_t>(row0 + r) * G + g);
        lane_dot<MT, WPL>(wd, xr, acc);
#pragma unroll
        for (int t = 0; t < MT; ++t) part[r][t] = acc[t] * s;
      } else {
#pragma unroll
        for (int t = 0; t < MT; ++t) part[r][t] = 0.f;
      }
    }
    float res[MT];
    warp_reduce_8rows<MT>(part, res, lane);
    float *redb = red + (c & 1) * nw * RC * MT;
    if ((lane & 3) == 0) {
      const int row = (lane >> 2) & 7;
#pragma unroll
      for (int t = 0; t < MT; ++t) redb[(warp * RC + row) * MT + t] = res[t];
    }
    named_bar_sync(1, blockDim.x);
    const bool abort = s_abort != 0;
    if (threadIdx.x == 0 && !abort && !p.fault && issued < nchunks) {
      issue(issued);
      ++issued;
    }
    if (threadIdx.x < RC * MT && !abort) {
      const int row = threadIdx.x / MT, t = threadIdx.x % MT;
      if (row < rows && t < p.mt) {
        float v = redb[row * MT + t];
        for (int w = 1; w < nw; ++w) v += redb[(w * RC + row) * MT + t];
        p.y[static_cast<size_t>(t) * p.ldy + row0 + row] = v;
      }
    }
    if (abort) break;
  }
  // After an abort, let copies already in flight land before the CTA exits.
  if (threadIdx.x == 0 && c < nchunks) {
    for (int d = c; d < issued; ++d) mbar_wait(&full[d % NS], static_cast<uint32_t>(d / NS) & 1u);
  }
}

template <int MT, int WPL, bool BF16>
cudaError_t launch_pass(const StreamParams &base, int N, int K, int nsm, int smem_optin,
                        bool overlap, cudaStream_t stream) {
  constexpr int SLICE = 32 * 8 * WPL;
  const int nw = (K + SLICE - 1) / SLICE;
  const int threads = nw * 32;
  StreamParams p = base;
  const uint32_t qrow = K / 2, srow = K / 8;
  const uint32_t stage = kRowsPerChunk * (qrow + (p.sc_bulk ? srow : 0));
  const size_t fixed = 2ull * nw * kRowsPerChunk * MT * sizeof(float) + 64;
  smem_optin -= 1024;  // room for the kernel's static shared memory
  const int chunks_per_sm = (N + nsm * kRowsPerChunk - 1) / (nsm * kRowsPerChunk);
  int ns = std::min(4, std::max(1, chunks_per_sm));
  while (ns > 1 && fixed + static_cast<size_t>(ns) * stage > static_cast<size_t>(smem_optin)) --ns;
  if (fixed + static_cast<size_t>(ns) * stage > static_cast<size_t>(smem_optin))
    return cudaErrorInvalidConfiguration;
  p.nstages = ns;
  const size_t smem = fixed + static_cast<size_t>(ns) * stage;
  auto kern = stream_gemm_kernel<MT, WPL, BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  int occ = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, threads, smem);
  if (e != cudaSuccess) return e;
  occ = std::max(occ, 1);
  const int grid = std::min((N + kRowsPerChunk - 1) / kRowsPerChunk, nsm * occ);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = overlap ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

int max_k_stream(int mt) { return mt == 1 ? 32 * 256 * 4 : 32 * 256; }

int stream_tile(int rem, int K) {
  // up to 4 tokens per pass; beyond K = 8192 one token per pass
  int mt = rem >= 3 ? 4 : rem;
  if (mt > 1 && K > max_k_stream(mt)) mt = 1;
  return mt;
}

int stream_gemm_passes(int M, int K) {
  int n = 0;
  for (int m0 = 0; m0 < M; ++n) m0 += std::min(stream_tile(M - m0, K), M - m0);
  return n;
}

cudaError_t launch_stream_gemm(const void *x, bool x_bf16, int ldx, const int32_t *qw,
                               const float *sc, int M, int N, int K, float *y, int ldy,
                               bool overlap, cudaStream_t stream) {
  const DeviceInfo &di = device_info();
  StreamParams base{};
  base.qw = qw;
  base.sc = sc;
  base.N = N;
  base.K = K;
  base.ldx = ldx;
  base.ldy = ldy;
  base.sc_bulk = (K % 128 == 0) ? 1 : 0;
  base.status = di.status;
  base.fault = take_injected_fault() ? 1 : 0;
  const size_t xb = x_bf16 ? 2 : 4;
  for (int m0 = 0; m0 < M;) {
    const int rem = M - m0;
    const int mt = stream_tile(rem, K);
    const int valid = std::min(mt, rem);
    StreamParams p = base;
    p.x = static_cast<const uint8_t *>(x) + static_cast<size_t>(m0) * ldx * xb;
    p.y = y + static_cast<size_t>(m0) * ldy;
    p.mt = valid;
    cudaError_t e;
    // lanes own one packed word per row (8 columns) when K allows, which
    // gives up to 32 warps per CTA to hide latency; 4 words beyond 8192
    if (mt == 1 && K <= 8192)
      e = x_bf16 ? launch_pass<1, 1, true>(p, N, K, di.num_sms, di.smem_optin, overlap, stream)
                 : launch_pass<1, 1, false>(p, N, K, di.num_sms, di.smem_optin, overlap, stream);
    else if (mt == 1)
      e = x_bf16 ? launch_pass<1, 4, true>(p, N, K, di.num_sms, di.smem_optin, overlap, stream)
                 : launch_pass<1, 4, false>(p, N, K, di.num_sms, di.smem_optin, overlap, stream);
    else if (mt == 2)
      e = x_bf16 ? launch_pass<2, 1, true>(p, N, K, di.num_sms, di.smem_optin, overlap, stream)
                 : launch_pass<2, 1, false>(p, N, K, di.num_sms, di.smem_optin, overlap, stream);
    else
      e = x_bf16 ? launch_pass<4, 2, true>(p, N, K, di.num_sms, di.smem_optin, overlap, stream)
                 : launch_pass<4, 2, false>(p, N, K, di.num_sms, di.smem_optin, overlap, stream);
    if (e != cudaSuccess) return e;
    m0 += valid;
  }
  return cudaSuccess;
}

}  // namespace w4a16
