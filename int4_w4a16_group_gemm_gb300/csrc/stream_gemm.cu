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
#include <cstdlib>
#include <mutex>

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

template <int MT, int WPL, bool BF16, bool SCB>
__global__ void __launch_bounds__(stream_max_threads(MT, WPL), 1)
    stream_gemm_kernel(const StreamParams p) {
  constexpr int EPL = 8 * WPL;
  constexpr int SLICE = 32 * EPL;
  constexpr int RC = kRowsPerChunk;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_abort;
  __shared__ int s_issued;

  const int K = p.K;
  const int nw = blockDim.x >> 5;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = K >> 5;
  const uint32_t qrow = static_cast<uint32_t>(K) >> 1;  // bytes per packed row
  const uint32_t srow = static_cast<uint32_t>(K) >> 3;  // bytes per scale row
  const uint32_t qstage = RC * qrow;
  const uint32_t stage_bytes = qstage + (SCB ? RC * srow : 0u);
  const int NS = p.nstages;

  // shared memory: NS stages | red[2][NS][nw][RC][MT] | count[2][NS] | full[NS]
  uint8_t *stages = smem;
  float *red = reinterpret_cast<float *>(smem + NS * stage_bytes);
  int *count = reinterpret_cast<int *>(red + 2 * NS * nw * RC * MT);
  uint64_t *full = reinterpret_cast<uint64_t *>(count + ((2 * NS + 1) & ~1));

  const int r0 = static_cast<int>((static_cast<long long>(p.N) * blockIdx.x) / gridDim.x);
  const int r1 = static_cast<int>((static_cast<long long>(p.N) * (blockIdx.x + 1)) / gridDim.x);
  const int nchunks = (r1 - r0 + RC - 1) / RC;

  auto issue = [&](int c) {
    const int slot = c % NS;
    const int row = r0 + c * RC;
    const int rows = min(RC, r1 - row);
    uint8_t *dst = stages + slot * stage_bytes;
    const uint32_t bq = rows * qrow;
    const uint32_t bs = SCB ? rows * srow : 0u;
    mbar_arrive_expect_tx(&full[slot], bq + bs);
    bulk_g2s(dst, reinterpret_cast<const uint8_t *>(p.qw) + static_cast<size_t>(row) * qrow, bq,
             &full[slot]);
    if (SCB)
      bulk_g2s(dst + qstage, reinterpret_cast<const uint8_t *>(p.sc) + static_cast<size_t>(row) * srow,
               bs, &full[slot]);
  };

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int i = 0; i < 2 * NS; ++i) count[i] = 0;
    for (int i = 0; i < NS; ++i) mbar_init(&full[i], 1);
    fence_mbar_init();
    // only the first stage before the activations: the SM serves its
    // requests roughly in order, and activations queued behind every
    // stage would arrive last
    const int first = p.fault ? 0 : min(1, nchunks);
    for (int c = 0; c < first; ++c) issue(c);
    s_issued = first;
  }
  __syncthreads();
  // The first weights are in flight. Let the next kernel start launching,
  // then wait for the previous one before touching x or y (both may be its
  // operands). Without programmatic launch both calls are no-ops.
  griddep_launch_dependents();
  griddep_wait();

  // This lane's columns and its activations (kept in registers).
  const int k0 = warp * SLICE + lane * EPL;
  const bool active = k0 < K;
  const int kc = active ? k0 : 0;  // inactive lanes read valid smem, weigh zero
  const int g = kc >> 5;
  uint64_t xr[MT][EPL / 2];
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
  // the activation loads are issued (their registers fill later); now the
  // remaining stages
  __syncthreads();
  if (threadIdx.x == 0 && !p.fault) {
    const int upto = min(NS, nchunks);
    for (int c = s_issued; c < upto; ++c) issue(c);
    s_issued = max(s_issued, upto);
  }

  for (int c = 0; c < nchunks; ++c) {
    const int slot = c % NS;
    const int half = (c / NS) & 1;
    const int row0 = r0 + c * RC;
    const int rows = min(RC, r1 - row0);
    // lane 0 waits for the stage (sleeping in hardware); __syncwarp then
    // orders the other lanes' reads after it
    int ok = 1;
    if (lane == 0) {
      ok = (s_abort == 0) && mbar_wait(&full[slot], static_cast<uint32_t>(c / NS) & 1u);
      if (!ok && s_abort == 0) {
        record_status(p.status, W4A16_ERR_TIMEOUT);
        s_abort = 1;
      }
    }
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    if (!ok) break;
    const uint8_t *st = stages + slot * stage_bytes;

    // 8 rows, branch-free: rows past the CTA's range hold stale bytes whose
    // sums are never stored
    float part[RC][MT];
    const uint8_t *wbase = st + (kc >> 1);
    // all 8 rows' words and scales first, so the loads overlap
    uint32_t wd[RC][WPL];
    float sv[RC];
#pragma unroll
    for (int r = 0; r < RC; ++r) {
      load_words<WPL>(wbase + r * qrow, wd[r]);
      sv[r] = SCB ? reinterpret_cast<const float *>(st + qstage + r * srow)[g]
                  : (r < rows ? __ldg(p.sc + static_cast<size_t>(row0 + r) * G + g) : 0.f);
    }
    rows_dot<MT, WPL>(wd, sv, xr, part);
    float res[MT];
    warp_reduce_8rows<MT>(part, res, lane);
    float *redc = red + (static_cast<size_t>(half * NS + slot) * nw) * RC * MT;
    if ((lane & 3) == 0) {
      const int row = (lane >> 2) & 7;
#pragma unroll
      for (int t = 0; t < MT; ++t) redc[(warp * RC + row) * MT + t] = res[t];
    }
    __syncwarp();
    int last = 0;
    if (lane == 0) {
      __threadfence_block();
      last = atomicAdd(&count[half * NS + slot], 1) == nw - 1;
    }
    last = __shfl_sync(0xFFFFFFFFu, last, 0);
    if (last) {
      // every warp has finished reading this stage: refill it first
      if (lane == 0) {
        __threadfence_block();
        count[half * NS + slot] = 0;
        if (c + NS < nchunks && s_abort == 0 && !p.fault) {
          issue(c + NS);
          atomicAdd(&s_issued, 1);
        }
      }
      __syncwarp();
      // fixed-order sum over the warps: lane (row r, part q) adds warps
      // q, q+4, q+8, ... in order, then the four parts pairwise
      const int r = lane >> 2, q = lane & 3;
#pragma unroll
      for (int t = 0; t < MT; ++t) {
        float v = 0.f;
        for (int w = q; w < nw; w += 4) v += redc[(w * RC + r) * MT + t];
        v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
        v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
        if (q == 0 && r < rows && t < p.mt) p.y[static_cast<size_t>(t) * p.ldy + row0 + r] = v;
      }
    }
  }
  // After an abort, let copies already in flight land before the CTA exits.
  __syncthreads();
  if (threadIdx.x == 0 && s_abort != 0) {
    for (int d = max(0, s_issued - NS); d < s_issued; ++d)
      mbar_wait(&full[d % NS], static_cast<uint32_t>(d / NS) & 1u);
  }
}

// Tuning overrides (read once): W4A16_STREAM_NS (stages, 1..8) and
// W4A16_STREAM_CTAS (CTAs per SM, 1..4); 0 = automatic.
int env_int(const char *name) {
  const char *v = getenv(name);
  return v ? atoi(v) : 0;
}

template <int MT, int WPL, bool BF16, bool SCB>
cudaError_t launch_pass(const StreamParams &base, int N, int K, int nsm, int smem_optin,
                        bool overlap, cudaStream_t stream) {
  constexpr int SLICE = 32 * 8 * WPL;
  const int nw = (K + SLICE - 1) / SLICE;
  const int threads = nw * 32;
  StreamParams p = base;
  const size_t stage = kRowsPerChunk * (K / 2 + (SCB ? K / 8 : 0));
  smem_optin -= 1024;  // room for the kernel's static shared memory
  static const int env_ns = env_int("W4A16_STREAM_NS");
  static const int env_ctas = env_int("W4A16_STREAM_CTAS");
  auto bytes_for = [&](int ns) {
    return static_cast<size_t>(ns) * stage + 2ull * ns * nw * kRowsPerChunk * MT * sizeof(float) +
           (2 * ns + 2) * sizeof(int) + ns * sizeof(uint64_t) + 64;
  };
  // Rows are split evenly over the grid. Each CTA's compute is bound by
  // instruction latency, so two CTAs per SM (each with up to 3 stages in
  // flight) stream faster than one with more stages; fall back to one CTA
  // per SM when two do not fit.
  int ctas_per_sm = env_ctas > 0 ? std::min(env_ctas, 4) : 2;
  const int rows_per_cta = (N + nsm * ctas_per_sm - 1) / (nsm * ctas_per_sm);
  const int want = std::max(1, (rows_per_cta + kRowsPerChunk - 1) / kRowsPerChunk);
  int ns = env_ns > 0 ? std::min(env_ns, 8) : std::min(ctas_per_sm > 1 ? 3 : 4, want);
  const size_t per_sm_budget = 227 * 1024;
  if (env_ctas <= 0 && ctas_per_sm > 1 && ctas_per_sm * (bytes_for(ns) + 1024) > per_sm_budget)
    ctas_per_sm = 1;
  while (ns > 1 && bytes_for(ns) > static_cast<size_t>(smem_optin)) --ns;
  if (bytes_for(ns) > static_cast<size_t>(smem_optin)) return cudaErrorInvalidConfiguration;
  p.nstages = ns;
  const size_t smem = bytes_for(ns);
  auto kern = stream_gemm_kernel<MT, WPL, BF16, SCB>;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin);
  });
  if (attr_err != cudaSuccess) return attr_err;
  // resident CTAs per SM for this configuration (cached for the last one)
  static std::mutex occ_mu;
  static size_t occ_smem = 0;
  static int occ_threads = 0, occ_val = 1;
  int occ;
  {
    std::lock_guard<std::mutex> lk(occ_mu);
    if (occ_smem != smem || occ_threads != threads) {
      int o = 0;
      cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kern, threads, smem);
      if (e != cudaSuccess) return e;
      occ_smem = smem;
      occ_threads = threads;
      occ_val = std::max(o, 1);
    }
    occ = occ_val;
  }
  const int grid = std::min((N + kRowsPerChunk - 1) / kRowsPerChunk,
                            nsm * std::min(occ, ctas_per_sm));
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

template <int MT, int WPL, bool BF16>
cudaError_t launch_pass_sc(const StreamParams &p, int N, int K, int nsm, int smem_optin,
                           bool overlap, cudaStream_t stream) {
  return p.sc_bulk ? launch_pass<MT, WPL, BF16, true>(p, N, K, nsm, smem_optin, overlap, stream)
                   : launch_pass<MT, WPL, BF16, false>(p, N, K, nsm, smem_optin, overlap, stream);
}

}  // namespace

int max_k_stream(int mt) { return mt == 1 ? 16384 : 8192; }

int stream_tile(int rem, int K) {
  // up to 3 tokens per pass (two packed words per lane, K <= 8192); one
  // token per pass (four words per lane) up to K = 16384
  const int mt = rem >= 3 ? 3 : rem;
  return K > max_k_stream(mt) ? 1 : mt;
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
    // one token: lanes own two packed words per row (16 columns) up to
    // K = 8192 (16 warps, 128 registers each), four beyond
    if (mt == 1 && K <= 8192)
      e = x_bf16 ? launch_pass_sc<1, 2, true>(p, N, K, di.num_sms, di.smem_optin, overlap, stream)
                 : launch_pass_sc<1, 2, false>(p, N, K, di.num_sms, di.smem_optin, overlap, stream);
    else if (mt == 1)
      e = x_bf16 ? launch_pass_sc<1, 4, true>(p, N, K, di.num_sms, di.smem_optin, overlap, stream)
                 : launch_pass_sc<1, 4, false>(p, N, K, di.num_sms, di.smem_optin, overlap, stream);
    else if (mt == 2)
      e = x_bf16 ? launch_pass_sc<2, 2, true>(p, N, K, di.num_sms, di.smem_optin, overlap, stream)
                 : launch_pass_sc<2, 2, false>(p, N, K, di.num_sms, di.smem_optin, overlap, stream);
    else
      e = x_bf16 ? launch_pass_sc<3, 2, true>(p, N, K, di.num_sms, di.smem_optin, overlap, stream)
                 : launch_pass_sc<3, 2, false>(p, N, K, di.num_sms, di.smem_optin, overlap, stream);
    if (e != cudaSuccess) return e;
    m0 += valid;
  }
  return cudaSuccess;
}

}  // namespace w4a16
