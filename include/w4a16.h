/*
 * w4a16.h - C ABI of the GB300 (sm_103a) W4A16 group-quantised GEMM library
 * (libw4a16.so).
 *
 * Weight format. "The Quiet Commit: How a Single Documentation Edit Marks the
 * Completion of a Major Engineering Milestone", section "The INT4 Milestone",
 * and section "Input Knowledge Required": symmetric per-group INT4 weights,
 * 8 nibbles packed per int32 along the input dimension (K), stored value
 * nibble = q + 8 (so the weight is nibble - 8), one fp32 scale per group of
 * `group` consecutive input columns: 32 is the size the pages fix; 64 and
 * 128 (the other common W4A16 group sizes) are taken too. Within a word,
 * input column k sits in bits 4*(k mod 8) .. 4*(k mod 8)+3 (low nibble
 * first).
 *   qw[N][K/8]      int32   row n = output feature, K-contiguous
 *   sc[N][K/group]  float   scale of (row n, group k/group)
 *   W_hat[n][k] = (nibble(n,k) - 8) * sc[n][k/group]
 *
 * Operation. "The Silence of Success: A Single Line That Speaks Volumes",
 * section "What the Edit Actually Built": activations (fp32; a bf16 mode
 * gives the 16-bit activations the W4A16 name stands for) times the INT4
 * weights with
 * fp32 accumulation:  y[m][n] = sum_k x[m][k] * W_hat[n][k]  ("NT": both
 * operands K-contiguous, y row-major fp32).
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the
 *     library never allocates, frees or retains them. Row-major, densely
 *     packed (leading dimension = row length) unless stated.
 *   - Calls are asynchronous on `stream` (NULL = legacy default stream).
 *     A return of W4A16_OK means the work was launched, not finished.
 *   - Argument errors are detected on the host before any launch and return
 *     a status without touching memory. Errors that depend on device data
 *     (an expert id outside [0, E)) or on a bounded device-side wait that
 *     ran out are recorded in a per-device status word; read and clear it
 *     with w4a16_last_device_status().
 *   - The library allocates nothing per call. The MoE entry point works in
 *     a caller-provided workspace whose size w4a16_moe_workspace_size()
 *     reports.
 *   - Results are deterministic: no floating-point atomics; every sum has a
 *     fixed order, so the same inputs give the same bits on every call.
 */
#ifndef W4A16_H_
#define W4A16_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* same type as cudaStream_t */
typedef struct CUstream_st *w4a16_stream_t;

typedef enum {
  W4A16_OK = 0,
  W4A16_ERR_INVALID_ARG = 1, /* null pointer, non-positive size, K not a
                                multiple of the group, bad enum, workspace
                                too small, id out of range */
  W4A16_ERR_UNSUPPORTED = 2, /* group not 32, 64 or 128, or a size beyond a
                                kernel limit */
  W4A16_ERR_ALIGNMENT = 3,   /* a pointer not 16-byte aligned */
  W4A16_ERR_CUDA = 4,        /* a CUDA runtime or launch error */
  W4A16_ERR_TIMEOUT = 5,     /* a bounded device-side wait ran out */
  W4A16_ERR_BOUNDS = 6       /* bounds-checking build only (compiled with
                                W4A16_DEBUG): a kernel computed an index
                                outside its buffer and skipped the access */
} w4a16_status;

typedef enum {
  W4A16_ACT_F32 = 0,  /* fp32 activations: the pages' kernel */
  W4A16_ACT_BF16 = 1  /* bf16 activations: the "A16" of W4A16 */
} w4a16_act_dtype;

/* Kernel choice for w4a16_gemm_ex (tests and tuning). */
typedef enum {
  W4A16_ALGO_AUTO = 0,   /* pick by M and dtype (what w4a16_gemm does) */
  W4A16_ALGO_SIMT = 1,   /* the streaming CUDA-core kernel, any M, both
                            dtypes (same as W4A16_ALGO_STREAM) */
  W4A16_ALGO_TC = 2,     /* tcgen05 tensor-core kernel: bf16 activations, or
                            fp32 activations with M <= 64 and K <= 16384
                            (each activation split exactly into three bf16
                            pieces, group scales applied in fp32) */
  W4A16_ALGO_STREAM = 3, /* the streaming CUDA-core kernel (token tiles of
                            up to 3), any M, K <= 16384 */
  W4A16_ALGO_GEMV = 4    /* the decode GEMV kernel: M = 1, K <= 8192 and
                            K/group a multiple of 4 (UNSUPPORTED otherwise).
                            One CTA per SM, sized so that under
                            W4A16_FLAG_OVERLAP the next call's CTA streams
                            its weights into shared memory beside it */
} w4a16_algo;

/*
 * w4a16_gemm - y = x * W_hat^T.
 *   x   [M][K]   fp32 or bf16 (xdt), device, 16-byte aligned
 *   qw  [N][K/8] int32 packed nibbles, device, 16-byte aligned
 *   sc  [N][K/group] fp32 scales, device, 16-byte aligned
 *   y   [M][N]   fp32 output, device, 16-byte aligned (overwritten)
 *   group is 32, 64 or 128; K a positive multiple of group; M, N > 0.
 * fp32 mode keeps every output within 1e-5 * sum_k |x*W_hat| of the exact
 * product; bf16 mode within 4e-3 of it (exact product of the bf16 values).
 * Kernels: bf16 with M >= 4 runs on the tensor cores; fp32 with
 * 12 <= M <= 64 on the tensor cores in the fp32-exact split form; the rest
 * on the streaming CUDA-core kernel.
 * Errors: INVALID_ARG, UNSUPPORTED (group not 32/64/128; K > 16384 on the CUDA-core
 * and fp32 tensor-core paths), ALIGNMENT, CUDA.
 */
w4a16_status w4a16_gemm(const void *x, w4a16_act_dtype xdt,
                        const int32_t *qw, const float *sc,
                        int M, int N, int K, int group,
                        float *y, w4a16_stream_t stream);

/* Launch options for w4a16_gemm_ex (bit flags). */
enum {
  /* Overlap with the previous kernel on the stream (programmatic dependent
   * launch): the call may begin streaming qw/sc while the kernel launched
   * just before it is still running; it reads x and writes y only after
   * that kernel has completed. The caller guarantees that the kernel
   * launched just before does not write qw or sc (true when weights are
   * prepared earlier, as in a decode loop). Every kernel honours it: the
   * tensor-core kernels dequantise their first stages of weights early. */
  W4A16_FLAG_OVERLAP = 1u,
  /* bf16 output: y is [M][N] bf16 (16-bit elements) instead of fp32; each
   * element is the fp32 result the same call would write without the flag,
   * rounded to nearest (ties to even). Halves the output bytes for callers
   * whose next layer consumes bf16. */
  W4A16_FLAG_OUT_BF16 = 2u
};

/* w4a16_gemm with an explicit kernel choice and launch flags (0 = none);
 * W4A16_ALGO_TC takes bf16 activations, or fp32 activations with M <= 64
 * and K <= 16384 (UNSUPPORTED otherwise). y is fp32 [M][N], or bf16
 * [M][N] with W4A16_FLAG_OUT_BF16 (16-byte aligned either way). Same
 * arguments and errors as w4a16_gemm, plus INVALID_ARG for unknown flags. */
w4a16_status w4a16_gemm_ex(const void *x, w4a16_act_dtype xdt,
                           const int32_t *qw, const float *sc,
                           int M, int N, int K, int group,
                           void *y, w4a16_algo algo, unsigned int flags,
                           w4a16_stream_t stream);

/* Number of kernel launches a w4a16_gemm_ex call with these arguments makes
 * (all on `stream`, in order), or -status if the call would be rejected.
 * Host-only; touches no device memory. */
int w4a16_gemm_launches(int M, int N, int K, int group, w4a16_act_dtype xdt,
                        w4a16_algo algo);

/*
 * w4a16_quantize - the per-group symmetric INT4 quantiser (the
 * quantize_w4a16 step of "The Quiet Commit: ... Major Engineering
 * Milestone", section "The INT4 Milestone"), to prepare weights on the
 * device:  s = max|w| / 7 (fp32 division), q = clamp(round-half-even(w / s),
 * -8, 7) (q = 0 when s = 0), nibble = q + 8, packed low nibble first.
 *   w  [N][K]    fp32 input (finite values), device
 *   qw [N][K/8]  int32 output, device;  sc [N][K/group] fp32 output, device
 *   group 32, 64 or 128; K a multiple of 32 and of group.
 * Errors: INVALID_ARG, UNSUPPORTED (group not 32/64/128), ALIGNMENT (qw or
 * w not 16-byte aligned), CUDA.
 */
w4a16_status w4a16_quantize(const float *w, int N, int K, int group,
                            int32_t *qw, float *sc, w4a16_stream_t stream);

/*
 * w4a16_moe_sort - group the (token, slot) pairs of a top-k routing by
 * expert, stably. Pair p = t*topk + slot, for p in [0, n_pairs).
 *   expert_ids [n_pairs] int32, device
 *   offsets    [E+1] int32 output: offsets[e] = number of pairs with an
 *              expert below e; offsets[E] = number of valid pairs
 *   perm       [n_pairs] int32 output: pairs ordered by (expert, p)
 * An id outside [0, E) is skipped and recorded as INVALID_ARG in the
 * device status word. One CTA; E <= 8192.
 */
w4a16_status w4a16_moe_sort(const int32_t *expert_ids, int n_pairs, int E,
                            int32_t *offsets, int32_t *perm,
                            w4a16_stream_t stream);

/* Bytes of workspace w4a16_moe_gemm needs for these sizes (either dtype). */
size_t w4a16_moe_workspace_size(int T, int topk, int E, int H, int I);

/* Where w4a16_moe_gemm leaves its intermediates in the workspace, for
 * inspection (per-stage checks and debugging); host-only. After a call
 * with these sizes the workspace holds, at the returned byte offsets:
 *   off_perm: perm [T*topk] int32, the pairs p = t*topk + slot in expert
 *             order (as w4a16_moe_sort returns it);
 *   off_h:    h [T*topk][I], row s = the SwiGLU output silu(g)*u of pair
 *             perm[s] - bf16 elements in bf16 mode, fp32 otherwise;
 *   off_o:    o [T*topk][H] fp32, row p = route_w[p] * (h @ W_hat_dn^T)
 *             of pair p (before the slot sum).
 * The same offsets hold for w4a16_moe_block, whose routed layer starts at
 * byte 0 of its workspace.
 * Errors: INVALID_ARG (non-positive size, null output pointer). */
w4a16_status w4a16_moe_workspace_layout(int T, int topk, int E, int H, int I,
                                        size_t *off_perm, size_t *off_h, size_t *off_o);

/*
 * w4a16_moe_gemm - a grouped MoE layer on INT4 experts ("The Quiet Commit:
 * ... Major Engineering Milestone", section "The Context: A Native DDTree
 * Engine Takes Shape" - MoE with SwiGLU - and section "The INT4 Milestone";
 * "The Quiet Commit: How a Single Plan Update Closed Phase 3 ...", section
 * "The Context: Phase 3 ..."):
 *   for each token t and slot j, e = expert_ids[t][j]:
 *     [g; u] = x[t] * W_hat_gu[e]^T   (g: rows 0..I-1, u: rows I..2I-1)
 *     h      = silu(g) * u            (stored as bf16 in bf16 mode)
 *     y[t]  += route_w[t][j] * (h * W_hat_dn[e]^T), slots summed in order.
 * Tokens are sorted by expert first, so each expert's weights are streamed
 * once per call whatever its token count.
 *   x        [T][H] fp32 or bf16 (xdt)
 *   expert_ids [T][topk] int32;  route_w [T][topk] fp32
 *   qw_gu [E][2I][H/8] int32;  sc_gu [E][2I][H/group] fp32
 *   qw_dn [E][H][I/8]  int32;  sc_dn [E][H][I/group]  fp32
 *   workspace: device memory of at least w4a16_moe_workspace_size() bytes,
 *   16-byte aligned, owned by the caller; contents on entry are ignored.
 *   y [T][H] fp32 output (overwritten).
 * group is 32, 64 or 128; H and I multiples of group, at most 16384.
 */
w4a16_status w4a16_moe_gemm(const void *x, w4a16_act_dtype xdt,
                            const int32_t *expert_ids, const float *route_w,
                            int T, int topk,
                            const int32_t *qw_gu, const float *sc_gu,
                            const int32_t *qw_dn, const float *sc_dn,
                            int E, int H, int I, int group,
                            void *workspace, size_t ws_bytes,
                            float *y, w4a16_stream_t stream);

/*
 * w4a16_moe_gemm_noalloc - w4a16_moe_gemm for callers that cannot allocate.
 * The pages have no counterpart to this entry point; it exists for host
 * code that may not allocate device memory once it is running (serving
 * processes that reserve their whole budget at start-up, plugins whose
 * host framework owns every allocation and offers no workspace, code where
 * a cudaMalloc would synchronise the device or take the allocator's lock).
 * It computes exactly what w4a16_moe_gemm computes, with the same
 * arguments minus the workspace, and calls no allocating routine.
 *   - Its intermediates live in one fixed device array inside the library:
 *     40 MiB (41943040 bytes), held by every GPU that loads the library
 *     until the process exits. Sizes whose w4a16_moe_workspace_size()
 *     exceeds it are rejected with W4A16_ERR_UNSUPPORTED before any work.
 *     (128 tokens x top-8, hidden 7168, expert width 2048 need ~37.4 MB.)
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first
 *     call before any stream capture on that device.
 *   - Every call shares the one array and leaves its contents behind; no
 *     intermediate needs to start at zero. Calls that overlap on the GPU
 *     (other streams, other host threads) race on it: order them.
 *   - The array used is the current device's: every pointer passed must be
 *     memory of the device that is current when the call is made.
 * Errors: as w4a16_moe_gemm, plus UNSUPPORTED for sizes beyond the array.
 */
w4a16_status w4a16_moe_gemm_noalloc(const void *x, w4a16_act_dtype xdt,
                                    const int32_t *expert_ids, const float *route_w,
                                    int T, int topk,
                                    const int32_t *qw_gu, const float *sc_gu,
                                    const int32_t *qw_dn, const float *sc_dn,
                                    int E, int H, int I, int group,
                                    float *y, w4a16_stream_t stream);

/*
 * w4a16_moe_route - the MoE router ("The Quiet Commit: ... Major Engineering
 * Milestone", section "The Context: A Native DDTree Engine Takes Shape", and
 * "The Quiet Commit: How a Single Plan Update Closed Phase 3 ...", section
 * "The Context: Phase 3 of a Custom Inference Stack": DeepSeekV3/Kimi-style
 * MoE routing; the pages give no formula, so the published DeepSeek-V3 gate
 * is used):
 *   logits[t][e] = x[t] . router_w[e]                  (fp32 accumulation)
 *   s = sigmoid(logits); expert_ids[t] = the topk experts with the largest
 *   s + router_bias, in decreasing order, equal values to the lower id;
 *   route_w[t][j] = route_scale * s[t][ids[t][j]] / sum_j' s[t][ids[t][j']].
 *   x [T][H] fp32 or bf16 (xdt), 16-byte aligned; H a multiple of 32
 *   router_w [E][H] fp32, 16-byte aligned; router_bias [E] fp32 or NULL
 *   logits [T][E] fp32, expert_ids [T][topk] int32, route_w [T][topk] fp32:
 *   outputs, caller-owned device memory (overwritten).
 * Errors: INVALID_ARG (null pointer, bad size, topk > E, route_scale not
 * finite), UNSUPPORTED (E > 1024 or topk > 32), ALIGNMENT, CUDA.
 */
w4a16_status w4a16_moe_route(const void *x, w4a16_act_dtype xdt, int T, int H,
                             const float *router_w, const float *router_bias, int E, int topk,
                             float route_scale, float *logits, int32_t *expert_ids,
                             float *route_w, w4a16_stream_t stream);

/* Bytes of workspace w4a16_moe_block needs (0 for invalid sizes); Is = 0
 * when there is no shared expert. */
size_t w4a16_moe_block_workspace_size(int T, int topk, int E, int H, int I, int Is);

/*
 * w4a16_moe_block - the whole MoE block on INT4 experts: router, routed
 * experts and the shared expert (same pages and sections as
 * w4a16_moe_route and w4a16_moe_gemm; "The INT4 Milestone": the shared
 * expert runs through the INT4 path too):
 *   route as w4a16_moe_route (ids and weights written to expert_ids and
 *   route_w), then
 *   y[t] = sum_j route_w[t][j] * expert_{ids[t][j]}(x[t]) + shared(x[t]),
 *   expert(x) = (silu(g) * u) * W_hat_dn^T with [g; u] = x * W_hat_gu^T
 *   (h = silu(g) * u stored as bf16 in bf16 mode), the shared expert added
 *   after the routed slots.
 *   Routed experts as w4a16_moe_gemm: qw_gu [E][2I][H/8], sc_gu
 *   [E][2I][H/group], qw_dn [E][H][I/8], sc_dn [E][H][I/group].
 *   Shared expert of width Is: qw_sgu [2Is][H/8], sc_sgu [2Is][H/group],
 *   qw_sdn [H][Is/8], sc_sdn [H][Is/group]; Is = 0 (pointers may be NULL)
 *   means no shared expert. Its two projections run as w4a16_gemm calls.
 *   workspace: at least w4a16_moe_block_workspace_size() bytes, 16-byte
 *   aligned, caller-owned; contents on entry are ignored.
 *   expert_ids [T][topk] int32, route_w [T][topk] fp32, y [T][H] fp32:
 *   outputs (overwritten); y 16-byte aligned.
 * group is 32, 64 or 128; H, I and Is multiples of group, at most 16384.
 * Errors: as w4a16_moe_route and w4a16_moe_gemm.
 */
w4a16_status w4a16_moe_block(const void *x, w4a16_act_dtype xdt, int T,
                             const float *router_w, const float *router_bias, int E, int topk,
                             float route_scale,
                             const int32_t *qw_gu, const float *sc_gu,
                             const int32_t *qw_dn, const float *sc_dn, int H, int I,
                             const int32_t *qw_sgu, const float *sc_sgu,
                             const int32_t *qw_sdn, const float *sc_sdn, int Is,
                             int group, void *workspace, size_t ws_bytes,
                             int32_t *expert_ids, float *route_w, float *y,
                             w4a16_stream_t stream);

/* Testing aid for failure detection: when `enable` is non-zero, the next
 * launch of a CUDA-core GEMM kernel (decode GEMV or streaming) on any device
 * skips issuing its weight copies, so its waits for them run out (after about one second) and it
 * records W4A16_ERR_TIMEOUT and returns. The switch clears itself after
 * that launch. No fault, trap or hang is involved; the context stays
 * usable. Not for production use. */
void w4a16_debug_fault_next_launch(int enable);

/* Human-readable name of a status code (static string). */
const char *w4a16_status_string(w4a16_status s);

/* Synchronises `stream`, then returns and clears the current device's status
 * word (OK if no kernel recorded an error since the last call). Returns
 * W4A16_ERR_CUDA if the synchronisation itself fails. */
w4a16_status w4a16_last_device_status(w4a16_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_H_ */
