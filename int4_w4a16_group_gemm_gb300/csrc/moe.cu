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
//               scatter of pair indices p = t*topk + slot (perm); the same
//               kernel lists the work items (expert, tile of up to MT of its
//               tokens) in expert order;
//  2. gate/up:  one CTA per (row block, work item): stream the block's gate
//               and up rows; h = silu(g) * u for the item's tokens, stored
//               per sorted position (bf16 in bf16 mode);
//  3. down:     the same over the down rows; o[p] = route_w[p] *
//               (h @ W_dn^T), stored per pair;
//  4. combine:  y[t] = o[t*topk + 0] + o[t*topk + 1] + ... (slot order),
//               plus the shared expert's output of token t when given.
// The work items of one expert are adjacent in the grid, so an expert's
// weights come from HBM once and from L2 for its further token tiles.
#include <algorithm>
#include <mutex>
#include <type_traits>

#include "kernels.h"
#include "stream_core.cuh"

namespace w4a16 {

namespace {

constexpr int kMaxExperts = 8192;

// ------------------------------------------------------------------ 1. sort
// Exclusive prefix sum of `v` over the block's threads (thread order);
// `scratch` holds 32 ints. Every thread of the block must call it.
__device__ int block_exclusive_scan(int v, int *scratch, int lane, int warp, int nt) {
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += u;
  }
  __syncthreads();  // scratch may still be read by a previous call
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int w = lane < (nt >> 5) ? scratch[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xFFFFFFFFu, wi, o);
      if (lane >= o) wi += u;
    }
    scratch[lane] = wi - w;  // exclusive prefix of warp totals
  }
  __syncthreads();
  return scratch[warp] + incl - v;
}

__global__ void __launch_bounds__(1024) moe_sort_kernel(const int32_t *__restrict__ ids, int n,
                                                        int E, int32_t *__restrict__ offsets,
                                                        int32_t *__restrict__ perm, int tile,
                                                        int32_t *__restrict__ items,
                                                        int32_t *__restrict__ n_items,
                                                        int *status) {
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
  // exclusive scans of cnt[0..E) and of the token tiles per expert: each
  // thread owns a contiguous chunk of experts
  const int per = (E + nt - 1) / nt;
  const int b = min(E, tid * per), f = min(E, b + per);
  int local = 0, local_t = 0;
  for (int e = b; e < f; ++e) {
    local += cnt[e];
    local_t += (cnt[e] + tile - 1) / tile;
  }
  const int lane = tid & 31, warp = tid >> 5;
  int run = block_exclusive_scan(local, warp_tot, lane, warp, nt);
  int item = block_exclusive_scan(local_t, warp_tot, lane, warp, nt);
  for (int e = b; e < f; ++e) {
    const int c = cnt[e];
    offsets[e] = run;
    cnt[e] = run;  // becomes the scatter cursor
    run += c;
    for (int j = 0; j * tile < c; ++j, ++item) {
      if (items != nullptr) {
        items[2 * item] = e;
        items[2 * item + 1] = j;
      }
    }
  }
  if (tid == nt - 1) {  // the last thread ends at the totals
    offsets[E] = run;
    if (n_items != nullptr) *n_items = item;
  }
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
  const void *x;          // gate/up: tokens [T][H]; down: h [n][I] (sorted order)
  const int32_t *perm;    // sorted position -> pair
  const int32_t *offsets;
  const int32_t *items;   // work items: (expert, token tile) pairs
  const int32_t *n_items;
  const float *route_w;   // [n]
  const int32_t *qw;      // expert-major packed weights
  const float *sc;
  void *out;              // gate/up: h [n][I]; down: o [n][H] fp32 (by pair)
  int H, I, topk;
  int n_pairs, E;  // buffer extents for the bounds-checking build
  int nstages;
  int gs;       // log2 of the group size
  int srow;     // bytes per scale row: (K / group) * 4, K the reduced dimension
  int sc_bulk;
  int *status;
};

// Rows of an expert per CTA: up to kMoeRowsPerCta (fewer per-CTA start-up
// and table costs; measured on the 128-token layer, 512 rows per CTA are 8%
// faster than 128), down to kMoeMinRowsPerCta while the grid would give the
// SMs fewer than 8 CTAs each (decode-sized calls with few work items, where
// smaller CTAs balance better: 4 tokens x top-8 measured 19% faster so).
constexpr int kMoeRowsPerCta = 512;
constexpr int kMoeMinRowsPerCta = 128;

// One CTA = one work item (an expert and a tile of up to MT of its tokens;
// blockIdx.x) x one block of the expert's rows (blockIdx.y). Consecutive
// CTAs take the tiles of one expert over the same rows, so those rows come
// from HBM once. The structure is the dense streaming
// kernel's: consumer warps own K-slices, the last warp streams 8-row stages
// into a ring with bulk copies and refills a stage as soon as every consumer
// has loaded its words, the per-warp row sums go to a table that the whole
// CTA adds in a fixed order at the end.
// MODE 0: gate/up (K = H). A stage holds 4 gate rows and the 4 matching up
//         rows; the epilogue writes h = silu(gate) * up.
// MODE 1: down (K = I), 8 rows per stage; the epilogue writes
//         o[pair] = route_w[pair] * (h @ W_dn^T).
template <int MT, int WPL, bool BF16, int MODE, int MAXW, int MINB>
__global__ void __launch_bounds__(32 * MAXW, MINB) moe_expert_kernel(const MoeParams p) {
  constexpr int EPL = 8 * WPL;
  constexpr int SLICE = 32 * EPL;
  constexpr int RC = kRowsPerChunk;
  constexpr int RL = MODE == 0 ? 4 : 8;  // logical output rows per stage
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_abort;

  const int it = blockIdx.x;
  if (it >= *p.n_items) return;  // the grid is sized for the most items
  const int e = p.items[2 * it];
  if (!W4A16_IN_BOUNDS(e >= 0 && e < p.E, p.status)) return;
  const int s0 = p.offsets[e] + p.items[2 * it + 1] * MT;
  const int mt = min(MT, p.offsets[e + 1] - s0);
  if (!W4A16_IN_BOUNDS(s0 >= 0 && s0 + mt <= p.n_pairs, p.status)) return;

  const int K = MODE == 0 ? p.H : p.I;
  const int L = MODE == 0 ? p.I : p.H;  // logical rows of the expert
  const int l_begin = static_cast<int>((static_cast<long long>(L) * blockIdx.y) / gridDim.y);
  const int l_end = static_cast<int>((static_cast<long long>(L) * (blockIdx.y + 1)) / gridDim.y);
  const int nchunks = (l_end - l_begin + RL - 1) / RL;

  const int nw = (blockDim.x >> 5) - 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t qrow = static_cast<uint32_t>(K) >> 1;
  const uint32_t srow = static_cast<uint32_t>(p.srow);
  const uint32_t qstage = RC * qrow;
  const uint32_t stage_bytes = qstage + (p.sc_bulk ? RC * srow : 0u);
  const int NS = p.nstages;
  const size_t erows = MODE == 0 ? 2 * static_cast<size_t>(p.I) : static_cast<size_t>(p.H);
  const uint8_t *qbase = reinterpret_cast<const uint8_t *>(p.qw) + e * erows * qrow;
  const uint8_t *sbase = reinterpret_cast<const uint8_t *>(p.sc) + e * erows * srow;

  // shared memory: NS stages | full[NS] | empty[NS] | red[nchunks*RC][MT][nw]
  uint8_t *stages = smem;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + NS * stage_bytes);
  uint64_t *empty = full + NS;
  float *red = reinterpret_cast<float *>(empty + NS);

  // expert row held by stage row r of chunk c (-1: past the block)
  auto stage_row = [&](int c, int r) -> int {
    const int l0 = l_begin + c * RL;
    if (MODE == 0) {
      const int j = l0 + (r & 3);
      if (j >= l_end) return -1;
      return r < 4 ? j : p.I + j;
    } else {
      const int n = l0 + r;
      return n < l_end ? n : -1;
    }
  };

  auto issue = [&](int c) {
    const int slot = c % NS;
    const int l0 = l_begin + c * RL;
    const int rows = min(RL, l_end - l0);
    uint8_t *dst = stages + slot * stage_bytes;
    const int parts = MODE == 0 ? 2 : 1;
    const uint32_t bq = rows * qrow, bs = p.sc_bulk ? rows * srow : 0u;
    // rows [l0, l0 + rows) (and the matching up rows) of this expert
    if (!W4A16_IN_BOUNDS(l0 >= 0 && rows > 0 && l0 + rows <= L, p.status))
      return;  // the stage never fills: its waits time out
    mbar_arrive_expect_tx(&full[slot], parts * (bq + bs));
    for (int h = 0; h < parts; ++h) {
      const size_t grow = static_cast<size_t>(l0) + (h ? p.I : 0);
      bulk_g2s(dst + h * 4 * qrow, qbase + grow * qrow, bq, &full[slot]);
      if (p.sc_bulk) bulk_g2s(dst + qstage + h * 4 * srow, sbase + grow * srow, bs, &full[slot]);
    }
  };

  const int first = min(NS, nchunks);
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

  if (warp == nw) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int issued = first, released = 0;
      for (int c = 0; c + NS < nchunks; ++c) {
        if (!mbar_wait_or_abort(&empty[c % NS], static_cast<uint32_t>(c / NS) & 1u, &s_abort)) {
          if (atomicExch(&s_abort, 1) == 0) record_status(p.status, W4A16_ERR_TIMEOUT);
          break;
        }
        released = c + 1;
        issue(c + NS);
        ++issued;
      }
      if (static_cast<volatile int &>(s_abort) != 0)
        for (int d = released; d < issued; ++d)
          mbar_wait(&full[d % NS], static_cast<uint32_t>(d / NS) & 1u);
    }
  } else {
    // ------------------------------------------------------------ consumers
    // The tile's token count selects the code path, so a tile of one or two
    // tokens does not pay for three.
    const NibbleConsts nk = make_nibble_consts();
    const int k0 = warp * SLICE + lane * EPL;
    const bool active = k0 < K;
    const int kc = active ? k0 : 0;
    const int g = kc >> p.gs;
    auto consume = [&](auto tokens) {
      constexpr int TM = decltype(tokens)::value;
      uint64_t xr[TM][EPL / 2];
#pragma unroll
      for (int t = 0; t < TM; ++t) {
        const void *row = nullptr;
        if (active && t < mt &&
            W4A16_IN_BOUNDS(k0 + EPL <= K && p.perm[s0 + t] >= 0 && p.perm[s0 + t] < p.n_pairs,
                            p.status)) {
          const int s = s0 + t;
          const size_t xrow = MODE == 0 ? static_cast<size_t>(p.perm[s] / p.topk) * p.H
                                        : static_cast<size_t>(s) * p.I;
          row = BF16 ? static_cast<const void *>(static_cast<const uint16_t *>(p.x) + xrow)
                     : static_cast<const void *>(static_cast<const float *>(p.x) + xrow);
        }
        load_x_slice<EPL, BF16>(row, k0, xr[t]);
      }
      for (int c = 0; c < nchunks; ++c) {
        const int slot = c % NS;
        float sv[RC];
        if (!p.sc_bulk) {
#pragma unroll
          for (int r = 0; r < RC; ++r) {
            const int grow = stage_row(c, r);
            sv[r] = grow >= 0 && W4A16_IN_BOUNDS(static_cast<size_t>(grow) < erows &&
                                                     g < (K >> p.gs),
                                                 p.status)
                        ? __ldg(reinterpret_cast<const float *>(
                                          sbase + static_cast<size_t>(grow) * srow) + g)
                              : 0.f;
          }
        }
        int ok = 1;
        if (lane == 0) {
          ok = mbar_wait_or_abort(&full[slot], static_cast<uint32_t>(c / NS) & 1u, &s_abort);
          if (!ok && atomicExch(&s_abort, 1) == 0) record_status(p.status, W4A16_ERR_TIMEOUT);
        }
        if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) break;
        const uint8_t *st = stages + slot * stage_bytes;
        const uint8_t *wbase = st + (kc >> 1);
        uint32_t wd[RC][WPL];
#pragma unroll
        for (int r = 0; r < RC; ++r) {
          load_words<WPL>(wbase + r * qrow, wd[r]);
          if (p.sc_bulk) sv[r] = reinterpret_cast<const float *>(st + qstage + r * srow)[g];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
        float part[RC][TM];
        rows_dot<TM, WPL>(wd, sv, xr, part, nk);
        float res[TM];
        warp_reduce_8rows<TM>(part, res, lane);
        if ((lane & 3) == 0) {
          const int row = c * RC + ((lane >> 2) & 7);
#pragma unroll
          for (int t = 0; t < TM; ++t) red[(row * MT + t) * nw + warp] = res[t];
        }
      }
    };
    if (MT >= 3 && mt >= 3)
      consume(std::integral_constant<int, (MT >= 3 ? 3 : 1)>{});
    else if (MT >= 2 && mt == 2)
      consume(std::integral_constant<int, (MT >= 2 ? 2 : 1)>{});
    else
      consume(std::integral_constant<int, 1>{});
  }

  // ------------------------------------------------------------ epilogue
  __syncthreads();
  if (static_cast<volatile int &>(s_abort) != 0) return;
  auto rowsum = [&](int prow, int t) {
    const float *v = red + static_cast<size_t>(prow * MT + t) * nw;
    float a = 0.f;
    for (int w = 0; w < nw; ++w) a += v[w];
    return a;
  };
  const int nl = l_end - l_begin;
  for (int i = threadIdx.x; i < nl * MT; i += blockDim.x) {
    const int l = i / MT, t = i - l * MT;
    if (t >= mt) continue;
    if (!W4A16_IN_BOUNDS(l_begin + l < L, p.status)) continue;
    if (MODE == 0) {
      const int prow = (l / 4) * RC + (l & 3);
      const float h = silu_f(rowsum(prow, t)) * rowsum(prow + 4, t);
      const size_t idx = static_cast<size_t>(s0 + t) * p.I + l_begin + l;
      if (BF16)
        static_cast<__nv_bfloat16 *>(p.out)[idx] = __float2bfloat16_rn(h);
      else
        static_cast<float *>(p.out)[idx] = h;
    } else {
      const int pair = p.perm[s0 + t];
      if (!W4A16_IN_BOUNDS(pair >= 0 && pair < p.n_pairs, p.status)) continue;
      static_cast<float *>(p.out)[static_cast<size_t>(pair) * p.H + l_begin + l] =
          p.route_w[pair] * rowsum(l, t);
    }
  }
}

// ------------------------------------------------------------------ 4. combine
__global__ void moe_combine_kernel(const float *__restrict__ o, const int32_t *__restrict__ ids,
                                   const float *__restrict__ shared, int T, int topk, int H,
                                   int E, float *__restrict__ y, int *status) {
  const int H4 = H >> 2;
  const long long total = static_cast<long long>(T) * H4;
  if (!W4A16_IN_BOUNDS(H % 4 == 0, status)) return;  // 16-byte rows
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
    if (shared != nullptr) {  // the shared expert: one more slot, weight 1
      const float4 v = reinterpret_cast<const float4 *>(shared + static_cast<size_t>(t) * H)[n4];
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    reinterpret_cast<float4 *>(y + static_cast<size_t>(t) * H)[n4] = acc;
  }
}

size_t align256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

struct WsLayout {
  size_t off_offsets, off_perm, off_items, off_nitems, off_h, off_o, total;
};

// Token tile of the expert kernels (the same for both, since the work items
// are listed once): 3 tokens with two packed words per lane while both K
// fit 15 consumer warps, else 1 token with four words per lane.
constexpr int kMoeKMultiToken = 15 * 512;
int moe_tile(int H, int I) { return (H <= kMoeKMultiToken && I <= kMoeKMultiToken) ? 3 : 1; }

int moe_max_items(int n, int E, int tile) { return (n + tile - 1) / tile + std::min(n, E); }

WsLayout ws_layout(int T, int topk, int E, int H, int I) {
  const size_t n = static_cast<size_t>(T) * topk;
  const int tile = moe_tile(H, I);
  WsLayout w{};
  w.off_offsets = 0;
  w.off_perm = align256(sizeof(int32_t) * (E + 1));
  w.off_items = w.off_perm + align256(sizeof(int32_t) * std::max<size_t>(n, 1));
  w.off_nitems = w.off_items +
                 align256(sizeof(int32_t) * 2 * std::max(1, moe_max_items(static_cast<int>(n), E, tile)));
  w.off_h = w.off_nitems + align256(sizeof(int32_t));
  w.off_o = w.off_h + align256(sizeof(float) * n * I);
  w.total = w.off_o + align256(sizeof(float) * n * H);
  return w;
}

template <int MT, int WPL, bool BF16, int MODE, int MAXW, int MINB>
cudaError_t launch_expert_kernel(MoeParams p, int K, int L, int max_items, const DeviceInfo &di,
                                 cudaStream_t stream) {
  constexpr int SLICE = 32 * 8 * WPL;
  const int nw = (K + SLICE - 1) / SLICE;
  if (nw + 1 > MAXW) return cudaErrorInvalidConfiguration;
  const int threads = (nw + 1) * 32;
  const int RL = MODE == 0 ? 4 : 8;
  // row blocks of kMoeMinRowsPerCta .. kMoeRowsPerCta weight rows
  const int phys = L * (kRowsPerChunk / RL);
  const int gx_few = (phys + kMoeRowsPerCta - 1) / kMoeRowsPerCta;
  const int gx_many = (phys + kMoeMinRowsPerCta - 1) / kMoeMinRowsPerCta;
  const int gx_fill = static_cast<int>((8LL * di.num_sms + max_items - 1) / std::max(1, max_items));
  const int gx = std::max(1, std::max(gx_few, std::min(gx_many, gx_fill)));
  const int lrows = (L + gx - 1) / gx;
  const int chunks = (lrows + RL - 1) / RL;
  const size_t stage = kRowsPerChunk * (K / 2 + (p.sc_bulk ? (K >> p.gs) * 4 : 0));
  const size_t table = static_cast<size_t>(chunks) * kRowsPerChunk * MT * nw * sizeof(float);
  const size_t budget = static_cast<size_t>(di.smem_optin) - 1024;
  auto bytes_for = [&](int ns) { return ns * stage + 2ull * ns * sizeof(uint64_t) + table; };
  int ns = std::min(3, chunks);
  while (ns > 1 && bytes_for(ns) > budget) --ns;
  if (bytes_for(ns) > budget) return cudaErrorInvalidConfiguration;
  p.nstages = ns;
  const size_t smem = bytes_for(ns);
  auto kern = moe_expert_kernel<MT, WPL, BF16, MODE, MAXW, MINB>;
  static PerDeviceOnce attr_once;
  const cudaError_t attr_err = attr_once.run([&] {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(budget));
  });
  if (attr_err != cudaSuccess) return attr_err;
  kern<<<dim3(max_items, gx), threads, smem, stream>>>(p);
  return cudaGetLastError();
}

template <int MODE>
cudaError_t launch_expert(MoeParams p, bool bf16, int tile, int max_items, const DeviceInfo &di,
                          cudaStream_t stream) {
  const int K = MODE == 0 ? p.H : p.I;
  const int L = MODE == 0 ? p.I : p.H;
  p.srow = (K >> p.gs) * 4;
  p.sc_bulk = ((K >> p.gs) % 4 == 0) ? 1 : 0;
  if (tile == 3)
    return bf16 ? launch_expert_kernel<3, 2, true, MODE, 16, 1>(p, K, L, max_items, di, stream)
                : launch_expert_kernel<3, 2, false, MODE, 16, 1>(p, K, L, max_items, di, stream);
  return bf16 ? launch_expert_kernel<1, 4, true, MODE, 17, 1>(p, K, L, max_items, di, stream)
              : launch_expert_kernel<1, 4, false, MODE, 17, 1>(p, K, L, max_items, di, stream);
}

}  // namespace

cudaError_t launch_moe_sort(const int32_t *ids, int n_pairs, int E, int32_t *offsets,
                            int32_t *perm, cudaStream_t stream) {
  const DeviceInfo &di = device_info();
  moe_sort_kernel<<<1, 1024, 0, stream>>>(ids, n_pairs, E, offsets, perm, 1, nullptr, nullptr,
                                          di.status);
  return cudaGetLastError();
}

size_t moe_workspace_bytes(int T, int topk, int E, int H, int I) {
  return ws_layout(T, topk, E, H, I).total;
}

void moe_workspace_offsets(int T, int topk, int E, int H, int I, size_t *off_perm, size_t *off_h,
                           size_t *off_o) {
  const WsLayout L = ws_layout(T, topk, E, H, I);
  *off_perm = L.off_perm;
  *off_h = L.off_h;
  *off_o = L.off_o;
}

cudaError_t launch_moe(const void *x, bool x_bf16, const int32_t *ids, const float *route_w,
                       int T, int topk, const int32_t *qw_gu, const float *sc_gu,
                       const int32_t *qw_dn, const float *sc_dn, int E, int H, int I,
                       int group, void *workspace, const float *shared_o, float *y,
                       cudaStream_t stream) {
  const DeviceInfo &di = device_info();
  const WsLayout L = ws_layout(T, topk, E, H, I);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  int32_t *offsets = reinterpret_cast<int32_t *>(ws + L.off_offsets);
  int32_t *perm = reinterpret_cast<int32_t *>(ws + L.off_perm);
  int32_t *items = reinterpret_cast<int32_t *>(ws + L.off_items);
  int32_t *n_items = reinterpret_cast<int32_t *>(ws + L.off_nitems);
  void *h = ws + L.off_h;
  float *o = reinterpret_cast<float *>(ws + L.off_o);
  const int n = T * topk;
  // bf16 activations at sizes the tensor-core expert kernels take: the same
  // sort with token tiles of 16, the activation rows gathered in sorted
  // order (into the o region, which the down GEMM overwrites afterwards),
  // then both expert GEMMs on the tensor cores (moe_tc.cu)
  if (x_bf16 && moe_tc_supported(n, H, I, group)) {
    const int tc_tile = 16;
    const int tc_items = moe_max_items(n, E, tc_tile);
    moe_sort_kernel<<<1, 1024, 0, stream>>>(ids, n, E, offsets, perm, tc_tile, items, n_items,
                                            di.status);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    uint16_t *xs = reinterpret_cast<uint16_t *>(o);
    err = launch_moe_gather(static_cast<const uint16_t *>(x), perm, n, topk, H, xs, stream);
    if (err != cudaSuccess) return err;
    err = launch_moe_tc(0, xs, qw_gu, sc_gu, offsets, items, n_items, perm, route_w, n, E, H, I,
                        group, tc_items, h, stream);
    if (err != cudaSuccess) return err;
    err = launch_moe_tc(1, static_cast<const uint16_t *>(h), qw_dn, sc_dn, offsets, items, n_items,
                        perm, route_w, n, E, H, I, group, tc_items, o, stream);
    if (err != cudaSuccess) return err;
    const long long work = static_cast<long long>(T) * (H / 4);
    const int grid = static_cast<int>(std::min<long long>((work + 255) / 256, di.num_sms * 8ll));
    moe_combine_kernel<<<std::max(grid, 1), 256, 0, stream>>>(o, ids, shared_o, T, topk, H, E, y,
                                                              di.status);
    return cudaGetLastError();
  }
  const int tile = moe_tile(H, I);
  const int max_items = moe_max_items(n, E, tile);

  moe_sort_kernel<<<1, 1024, 0, stream>>>(ids, n, E, offsets, perm, tile, items, n_items,
                                          di.status);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;

  MoeParams p{};
  p.perm = perm;
  p.offsets = offsets;
  p.items = items;
  p.n_items = n_items;
  p.route_w = route_w;
  p.H = H;
  p.I = I;
  p.topk = topk;
  p.n_pairs = n;
  p.E = E;
  p.gs = group == 128 ? 7 : group == 64 ? 6 : 5;
  p.status = di.status;

  p.x = x;
  p.qw = qw_gu;
  p.sc = sc_gu;
  p.out = h;
  err = launch_expert<0>(p, x_bf16, tile, max_items, di, stream);
  if (err != cudaSuccess) return err;

  p.x = h;
  p.qw = qw_dn;
  p.sc = sc_dn;
  p.out = o;
  err = launch_expert<1>(p, x_bf16, tile, max_items, di, stream);
  if (err != cudaSuccess) return err;

  const long long work = static_cast<long long>(T) * (H / 4);
  const int grid = static_cast<int>(std::min<long long>((work + 255) / 256, di.num_sms * 8ll));
  moe_combine_kernel<<<std::max(grid, 1), 256, 0, stream>>>(o, ids, shared_o, T, topk, H, E, y,
                                                            di.status);
  return cudaGetLastError();
}

}  // namespace w4a16
