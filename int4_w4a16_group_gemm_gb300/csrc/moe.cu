// Grouped MoE layer on INT4 experts.
//
// "The Quiet Commit: How a Single Documentation Edit Marks the Completion of
// a Major Engineering Milestone", section "The Context: A Native DDTree
// Engine Takes Shape" (MoE experts with SwiGLU) and section "The INT4
// Milestone" (experts run through the W4A16 kernel); "The Quiet Commit: How
// a Single Plan Update Closed Phase 3 of a Native DDTree Inference Engine",
// section "The Context: Phase 3 ..." (the INT4 W4A16 group-quantised MoE
// path).
//
// Steps, all on the device and on one stream (the host reads nothing back):
//  1. sort:     histogram of expert ids -> exclusive scan (offsets) -> stable
//               scatter of pair indices p = t*topk + slot (perm);
//  2. gate/up:  per expert, stream its gate and up rows once; every token of
//               the expert multiplies them; h = silu(g) * u, stored per
//               sorted position (bf16 in bf16 mode);
//  3. down:     per expert, stream its down rows once; o[p] = route_w[p] *
//               (h @ W_dn^T), stored per pair;
//  4. combine:  y[t] = o[t*topk + 0] + o[t*topk + 1] + ... (slot order).
// Each expert's weights are read once per call whatever its token count.
#include <algorithm>
#include <mutex>

#include "kernels.h"
#include "stream_core.cuh"

namespace w4a16 {

namespace {

constexpr int kMaxExperts = 8192;

// ------------------------------------------------------------------ 1. sort
__global__ void __launch_bounds__(1024) moe_sort_kernel(const int32_t *__restrict__ ids, int n,
                                                        int E, int32_t *__restrict__ offsets,
                                                        int32_t *__restrict__ perm, int *status) {
  __shared__ int cnt[kMaxExperts];
  __shared__ int warp_tot[32];
  const int tid = threadIdx.x, nt = blockDim.x;
  for (int e = tid; e < E; e += nt) cnt[e] = 0;
  __syncthreads();
  for (int p = tid; p < n; p += nt) {
    const int e = ids[p];
    if (e >= 0 && e < E)
      atomicAdd(&cnt[e], 1);
    else
      record_status(status, W4A16_ERR_INVALID_ARG);
  }
  __syncthreads();
  // exclusive scan of cnt[0..E): each thread owns a contiguous chunk
  const int per = (E + nt - 1) / nt;
  const int b = min(E, tid * per), f = min(E, b + per);
  int local = 0;
  for (int e = b; e < f; ++e) local += cnt[e];
  const int lane = tid & 31, warp = tid >> 5;
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < (nt >> 5) ? warp_tot[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, wi, o);
      if (lane >= o) wi += v;
    }
    warp_tot[lane] = wi - w;  // exclusive prefix of warp totals
  }
  __syncthreads();
  int run = warp_tot[warp] + incl - local;
  for (int e = b; e < f; ++e) {
    const int c = cnt[e];
    offsets[e] = run;
    cnt[e] = run;  // becomes the scatter cursor
    run += c;
  }
  if (tid == nt - 1) offsets[E] = run;  // last thread ends at the total
  __syncthreads();
  // stable scatter by warp 0, 32 pairs at a time in pair order
  if (warp == 0) {
    const unsigned lt = (1u << lane) - 1u;
    for (int base = 0; base < n; base += 32) {
      const int p = base + lane;
      const bool in = p < n;
      int e = in ? ids[p] : -1;
      const bool valid = in && e >= 0 && e < E;
      if (!valid) e = -1 - lane;  // unique key: never matches a valid id
      const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
      int pos = 0;
      if (valid) pos = cnt[e] + __popc(peers & lt);
      __syncwarp();
      if (valid) {
        perm[pos] = p;
        if ((peers & lt) == 0) cnt[e] += __popc(peers);
      }
      __syncwarp();
    }
  }
}

// --------------------------------------------------------- 2./3. expert GEMMs
struct MoeParams {
  const void *x;        // gate/up: tokens [T][H]; down: h [n][I] (sorted order)
  const int32_t *perm;  // sorted position -> pair
  const int32_t *offsets;
  const float *route_w;  // [n]
  const int32_t *qw;     // expert-major packed weights
  const float *sc;
  void *out;             // gate/up: h [n][I]; down: o [n][H] fp32 (by pair)
  int H, I, topk;
  int nstages;
  int sc_bulk;
  int *status;
};

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

// MODE 0: gate/up + SwiGLU (K = H; a stage holds 4 gate rows and the 4
//         matching up rows, giving 4 columns of h).
// MODE 1: down + routing weight (K = I; 8 rows of the down projection).
// A CTA owns expert blockIdx.y and a range of its stages; the expert's
// tokens are taken in tiles of MT, and every resident stage serves up to
// kMoeTiles tiles before it is refilled, so an expert's weights stream from
// HBM once for up to kMoeTiles * MT tokens (more tokens: further passes).
// Within a pass the structure is the dense streaming kernel's: bulk copies
// into a ring of stages, 8 rows per stage, and the last warp to finish a
// stage refills it and reduces the warps' partial sums in a fixed order.
constexpr int kMoeTiles = 4;

template <int MT, int WPL, bool BF16, int MODE>
__global__ void __launch_bounds__(stream_max_threads(MT, WPL), 1) moe_stream_kernel(const MoeParams p) {
  constexpr int EPL = 8 * WPL;
  constexpr int SLICE = 32 * EPL;
  constexpr int RC = kRowsPerChunk;
  constexpr int RL = MODE == 0 ? 4 : 8;  // logical output rows per stage
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_abort;
  __shared__ int s_issued;

  const int e = blockIdx.y;
  const int s0 = p.offsets[e];
  const int ce = p.offsets[e + 1] - s0;
  if (ce <= 0) return;

  const int K = MODE == 0 ? p.H : p.I;
  const int L = MODE == 0 ? p.I : p.H;  // logical rows of the expert
  const int nlc = (L + RL - 1) / RL;
  const int c_begin = static_cast<int>((static_cast<long long>(nlc) * blockIdx.x) / gridDim.x);
  const int c_end = static_cast<int>((static_cast<long long>(nlc) * (blockIdx.x + 1)) / gridDim.x);
  const int nchunks = c_end - c_begin;
  if (nchunks <= 0) return;
  const int ntiles = (ce + MT - 1) / MT;
  const int npass = (ntiles + kMoeTiles - 1) / kMoeTiles;
  const int total = nchunks * npass;  // stages over all passes

  const int nw = blockDim.x >> 5;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = K >> 5;
  const uint32_t qrow = static_cast<uint32_t>(K) >> 1;
  const uint32_t srow = static_cast<uint32_t>(K) >> 3;
  const uint32_t qstage = RC * qrow;
  const uint32_t stage_bytes = qstage + (p.sc_bulk ? RC * srow : 0u);
  const int NS = p.nstages;
  const size_t erows = MODE == 0 ? 2 * static_cast<size_t>(p.I) : static_cast<size_t>(p.H);
  const uint8_t *qbase = reinterpret_cast<const uint8_t *>(p.qw) + e * erows * qrow;
  const uint8_t *sbase = reinterpret_cast<const uint8_t *>(p.sc) + e * erows * srow;

  uint8_t *stages = smem;
  float *red = reinterpret_cast<float *>(smem + NS * stage_bytes);
  int *count = reinterpret_cast<int *>(red + 2 * NS * kMoeTiles * nw * RC * MT);
  uint64_t *full = reinterpret_cast<uint64_t *>(count + ((2 * NS + 1) & ~1));

  // global row of stage row r for logical chunk starting at l0 (-1: none)
  auto stage_row = [&](int l0, int r) -> int {
    if (MODE == 0) {
      const int j = l0 + (r & 3);
      if (j >= p.I) return -1;
      return r < 4 ? j : p.I + j;
    } else {
      const int n = l0 + r;
      return n < p.H ? n : -1;
    }
  };

  auto issue = [&](int gc) {  // gc: stage index over all passes
    const int slot = gc % NS;
    const int l0 = (c_begin + gc % nchunks) * RL;
    const int rows = min(RL, L - l0);
    uint8_t *dst = stages + slot * stage_bytes;
    const int parts = MODE == 0 ? 2 : 1;
    const uint32_t bq = rows * qrow, bs = p.sc_bulk ? rows * srow : 0u;
    mbar_arrive_expect_tx(&full[slot], parts * (bq + bs));
    for (int h = 0; h < parts; ++h) {
      const size_t grow = static_cast<size_t>(l0) + (h ? p.I : 0);
      bulk_g2s(dst + h * 4 * qrow, qbase + grow * qrow, bq, &full[slot]);
      if (p.sc_bulk) bulk_g2s(dst + qstage + h * 4 * srow, sbase + grow * srow, bs, &full[slot]);
    }
  };

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int i = 0; i < 2 * NS; ++i) count[i] = 0;
    for (int i = 0; i < NS; ++i) mbar_init(&full[i], 1);
    fence_mbar_init();
    const int first = min(NS, total);
    for (int gc = 0; gc < first; ++gc) issue(gc);
    s_issued = first;
  }
  __syncthreads();

  const NibbleConsts nk = make_nibble_consts();
  const int k0 = warp * SLICE + lane * EPL;
  const bool active = k0 < K;
  const int kc = active ? k0 : 0;
  const int g = kc >> 5;

  uint64_t xr[MT][EPL / 2];
  auto load_tile = [&](int tile) {
#pragma unroll
    for (int t = 0; t < MT; ++t) {
      const int q = tile * MT + t;
      const void *row = nullptr;
      if (active && q < ce) {
        const int s = s0 + q;
        if (MODE == 0) {
          const int tok = p.perm[s] / p.topk;
          row = BF16 ? static_cast<const void *>(static_cast<const uint16_t *>(p.x) +
                                                 static_cast<size_t>(tok) * p.H)
                     : static_cast<const void *>(static_cast<const float *>(p.x) +
                                                 static_cast<size_t>(tok) * p.H);
        } else {
          row = BF16 ? static_cast<const void *>(static_cast<const uint16_t *>(p.x) +
                                                 static_cast<size_t>(s) * p.I)
                     : static_cast<const void *>(static_cast<const float *>(p.x) +
                                                 static_cast<size_t>(s) * p.I);
        }
      }
      load_x_slice<EPL, BF16>(row, k0, xr[t]);
    }
  };

  for (int gc = 0; gc < total; ++gc) {
    const int pass = gc / nchunks;
    const int c = gc % nchunks;
    const int t_begin = pass * kMoeTiles;
    const int nt = min(kMoeTiles, ntiles - t_begin);
    if (nt == 1 && c == 0) load_tile(t_begin);  // single tile: x stays in registers
    const int slot = gc % NS;
    const int half = (gc / NS) & 1;
    const int l0 = (c_begin + c) * RL;
    int ok = 1;
    if (lane == 0) {
      ok = (s_abort == 0) && mbar_wait(&full[slot], static_cast<uint32_t>(gc / NS) & 1u);
      if (!ok && s_abort == 0) {
        record_status(p.status, W4A16_ERR_TIMEOUT);
        s_abort = 1;
      }
    }
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    if (!ok) break;
    const uint8_t *st = stages + slot * stage_bytes;
    const uint8_t *wbase = st + (kc >> 1);
    float *redc = red + (static_cast<size_t>(half * NS + slot) * kMoeTiles) * nw * RC * MT;
#pragma unroll 1
    for (int j = 0; j < nt; ++j) {
      if (nt > 1) load_tile(t_begin + j);
      // the stage's words and scales, read per tile so that nothing but the
      // activations stays live across tiles
      uint32_t wd[RC][WPL];
      float sv[RC];
#pragma unroll
      for (int r = 0; r < RC; ++r) {
        load_words<WPL>(wbase + r * qrow, wd[r]);
        const int grow = stage_row(l0, r);
        sv[r] = p.sc_bulk ? reinterpret_cast<const float *>(st + qstage + r * srow)[g]
                          : (grow >= 0 ? __ldg(reinterpret_cast<const float *>(sbase) +
                                               static_cast<size_t>(grow) * G + g)
                                       : 0.f);
      }
      float part[RC][MT];
      rows_dot<MT, WPL>(wd, sv, xr, part, nk);
      float res[MT];
      warp_reduce_8rows<MT>(part, res, lane);
      if ((lane & 3) == 0) {
        const int row = (lane >> 2) & 7;
#pragma unroll
        for (int t = 0; t < MT; ++t) redc[((j * nw + warp) * RC + row) * MT + t] = res[t];
      }
    }
    __syncwarp();
    int last = 0;
    if (lane == 0) {
      __threadfence_block();
      last = atomicAdd(&count[half * NS + slot], 1) == nw - 1;
    }
    last = __shfl_sync(0xFFFFFFFFu, last, 0);
    if (!last) continue;
    // every warp has finished reading this stage: refill it first
    if (lane == 0) {
      __threadfence_block();
      count[half * NS + slot] = 0;
      if (gc + NS < total && s_abort == 0) {
        issue(gc + NS);
        atomicAdd(&s_issued, 1);
      }
    }
    __syncwarp();
    // fixed-order sum over the warps: lane (row r, part q) adds warps
    // q, q+4, ... in order, then the four parts pairwise
    const int r = lane >> 2, q = lane & 3;
    for (int j = 0; j < nt; ++j) {
      const int tile = t_begin + j;
      float v[MT];
#pragma unroll
      for (int t = 0; t < MT; ++t) {
        float a = 0.f;
        for (int w = q; w < nw; w += 4) a += redc[((j * nw + w) * RC + r) * MT + t];
        a += __shfl_xor_sync(0xFFFFFFFFu, a, 1);
        a += __shfl_xor_sync(0xFFFFFFFFu, a, 2);
        v[t] = a;
      }
      if (MODE == 0) {
        // lanes of rows 0-3 hold the gate sums, rows 4-7 the up sums
#pragma unroll
        for (int t = 0; t < MT; ++t) {
          const float up = __shfl_down_sync(0xFFFFFFFFu, v[t], 16);
          const int tq = tile * MT + t;
          if (q == 0 && r < 4 && l0 + r < p.I && tq < ce) {
            const float h = silu_f(v[t]) * up;
            const size_t idx = static_cast<size_t>(s0 + tq) * p.I + l0 + r;
            if (BF16)
              static_cast<__nv_bfloat16 *>(p.out)[idx] = __float2bfloat16_rn(h);
            else
              static_cast<float *>(p.out)[idx] = h;
          }
        }
      } else {
#pragma unroll
        for (int t = 0; t < MT; ++t) {
          const int tq = tile * MT + t;
          if (q == 0 && l0 + r < p.H && tq < ce) {
            const int pair = p.perm[s0 + tq];
            static_cast<float *>(p.out)[static_cast<size_t>(pair) * p.H + l0 + r] =
                p.route_w[pair] * v[t];
          }
        }
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && s_abort != 0) {
    for (int d = max(0, s_issued - NS); d < s_issued; ++d)
      mbar_wait(&full[d % NS], static_cast<uint32_t>(d / NS) & 1u);
  }
}

// ------------------------------------------------------------------ 4. combine
__global__ void moe_combine_kernel(const float *__restrict__ o, const int32_t *__restrict__ ids,
                                   int T, int topk, int H, int E, float *__restrict__ y) {
  const int H4 = H >> 2;
  const long long total = static_cast<long long>(T) * H4;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(i / H4);
    const int n4 = static_cast<int>(i % H4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < topk; ++j) {
      const int pair = t * topk + j;
      const int e = ids[pair];
      if (e < 0 || e >= E) continue;
      const float4 v = reinterpret_cast<const float4 *>(o + static_cast<size_t>(pair) * H)[n4];
      if (j == 0) {
        acc = v;
      } else {
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
      }
    }
    reinterpret_cast<float4 *>(y + static_cast<size_t>(t) * H)[n4] = acc;
  }
}

size_t align256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

struct WsLayout {
  size_t off_offsets, off_perm, off_h, off_o, total;
};

WsLayout ws_layout(int T, int topk, int E, int H, int I) {
  const size_t n = static_cast<size_t>(T) * topk;
  WsLayout w{};
  w.off_offsets = 0;
  w.off_perm = align256(sizeof(int32_t) * (E + 1));
  w.off_h = w.off_perm + align256(sizeof(int32_t) * std::max<size_t>(n, 1));
  w.off_o = w.off_h + align256(sizeof(float) * n * I);
  w.total = w.off_o + align256(sizeof(float) * n * H);
  return w;
}

template <int MT, int WPL, bool BF16, int MODE>
cudaError_t launch_expert_pass(MoeParams p, int K, int E, const DeviceInfo &di,
                               cudaStream_t stream) {
  constexpr int SLICE = 32 * 8 * WPL;
  const int nw = (K + SLICE - 1) / SLICE;
  const int threads = nw * 32;
  const size_t stage = kRowsPerChunk * (K / 2 + (p.sc_bulk ? K / 8 : 0));
  const size_t budget = static_cast<size_t>(di.smem_optin) - 1024;
  auto bytes_for = [&](int ns) {
    return static_cast<size_t>(ns) * stage +
           2ull * ns * kMoeTiles * nw * kRowsPerChunk * MT * sizeof(float) +
           (2 * ns + 2) * sizeof(int) + ns * sizeof(uint64_t) + 64;
  };
  // three stages keep two CTAs per SM resident for the widest experts
  int ns = 3;
  while (ns > 1 && bytes_for(ns) > budget) --ns;
  if (bytes_for(ns) > budget) return cudaErrorInvalidConfiguration;
  p.nstages = ns;
  const size_t smem = bytes_for(ns);
  auto kern = moe_stream_kernel<MT, WPL, BF16, MODE>;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(budget));
  });
  if (attr_err != cudaSuccess) return attr_err;
  // split every expert into several CTAs so the active experts spread
  // evenly over the SMs (empty experts exit at once)
  const int per_expert = 8;
  dim3 grid(per_expert, E);
  kern<<<grid, threads, smem, stream>>>(p);
  return cudaGetLastError();
}

template <int MODE>
cudaError_t launch_expert(MoeParams p, bool bf16, int K, int E, const DeviceInfo &di,
                          cudaStream_t stream) {
  p.sc_bulk = (K % 128 == 0) ? 1 : 0;
  // token tiles of 3 (bf16) or 2 (fp32, whose wider activation registers
  // would not fit 3) with two packed words per lane up to K = 8192
  if (K <= max_k_stream(3))
    return bf16 ? launch_expert_pass<3, 2, true, MODE>(p, K, E, di, stream)
                : launch_expert_pass<2, 2, false, MODE>(p, K, E, di, stream);
  return bf16 ? launch_expert_pass<1, 4, true, MODE>(p, K, E, di, stream)
              : launch_expert_pass<1, 4, false, MODE>(p, K, E, di, stream);
}

}  // namespace

cudaError_t launch_moe_sort(const int32_t *ids, int n_pairs, int E, int32_t *offsets,
                            int32_t *perm, cudaStream_t stream) {
  const DeviceInfo &di = device_info();
  moe_sort_kernel<<<1, 1024, 0, stream>>>(ids, n_pairs, E, offsets, perm, di.status);
  return cudaGetLastError();
}

size_t moe_workspace_bytes(int T, int topk, int E, int H, int I) {
  return ws_layout(T, topk, E, H, I).total;
}

cudaError_t launch_moe(const void *x, bool x_bf16, const int32_t *ids, const float *route_w,
                       int T, int topk, const int32_t *qw_gu, const float *sc_gu,
                       const int32_t *qw_dn, const float *sc_dn, int E, int H, int I,
                       void *workspace, float *y, cudaStream_t stream) {
  const DeviceInfo &di = device_info();
  const WsLayout L = ws_layout(T, topk, E, H, I);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  int32_t *offsets = reinterpret_cast<int32_t *>(ws + L.off_offsets);
  int32_t *perm = reinterpret_cast<int32_t *>(ws + L.off_perm);
  void *h = ws + L.off_h;
  float *o = reinterpret_cast<float *>(ws + L.off_o);
  const int n = T * topk;

  cudaError_t err = launch_moe_sort(ids, n, E, offsets, perm, stream);
  if (err != cudaSuccess) return err;

  MoeParams p{};
  p.perm = perm;
  p.offsets = offsets;
  p.route_w = route_w;
  p.H = H;
  p.I = I;
  p.topk = topk;
  p.status = di.status;

  p.x = x;
  p.qw = qw_gu;
  p.sc = sc_gu;
  p.out = h;
  err = launch_expert<0>(p, x_bf16, H, E, di, stream);
  if (err != cudaSuccess) return err;

  p.x = h;
  p.qw = qw_dn;
  p.sc = sc_dn;
  p.out = o;
  err = launch_expert<1>(p, x_bf16, I, E, di, stream);
  if (err != cudaSuccess) return err;

  const long long work = static_cast<long long>(T) * (H / 4);
  const int grid = static_cast<int>(std::min<long long>((work + 255) / 256, di.num_sms * 8ll));
  moe_combine_kernel<<<std::max(grid, 1), 256, 0, stream>>>(o, ids, T, topk, H, E, y);
  return cudaGetLastError();
}

}  // namespace w4a16
