"""CPU oracle for the W4A16 group-quantised GEMM and its grouped-MoE variant.

TEST INFRASTRUCTURE ONLY. The CUDA library never imports, links or runs this
package; only the tests, the smoke check and the benchmark's CPU-baseline leg
do. It shares no code with the CUDA path: both take their inputs from the
``synth`` random-draw module and nothing else.

It is the plain definition of what the path computes, in numpy, accumulated
in fp64 (a library matmul serves as the dot-product step). Sources, by page
title and section:

[SoS]  "The Silence of Success: A Single Line That Speaks Volumes"
       - "What the Edit Actually Built": fp32 activations times 4-bit weights
         packed two per byte, one scale per group of 32 input columns.
       - "The Weight of Context" / "Assumptions Embedded in the Code": the
         golden result is the dequantise-then-multiply product; fp32
         accumulation; group 32 must divide K.
[QC]   "The Quiet Commit: How a Single Documentation Edit Marks the
       Completion of a Major Engineering Milestone"
       - "The INT4 Milestone": symmetric quantisation, 8 nibbles per int32
         along the input dimension, value = nibble - 8, fp32 per-group
         scales (``quantize_w4a16``), packed ``.qw`` int32 and ``.sc`` fp32
         tensors, goldens computed from the dequantised weights.
       - "Input Knowledge Required": group size 32, value = nibble - 8.
       - "The Context: A Native DDTree Engine Takes Shape": MoE experts with
         SwiGLU between the gate/up and down projections.
[PC]   "The Quiet Commit: How a Single Plan Update Closed Phase 3 of a
       Native DDTree Inference Engine" - "The Context: Phase 3 ...": the
       INT4 W4A16 group-quantised MoE path.

Readings where the pages are silent (each is listed in the design notes):
  * nibble order inside the int32: low nibble first (k mod 8 = 0 in bits 0-3);
  * quantiser: s = max|w| / 7 in fp32, q = clamp(rne(w / s), -8, 7) with an
    fp32 division, nibble = q + 8; an all-zero group has s = 0 and q = 0;
  * dequantised weight: fp32 product (nibble - 8) * s;
  * bf16 activation mode: the caller's bf16 values are the activations;
  * MoE: gate rows 0..I-1 and up rows I..2I-1 of the fused gate+up matrix,
    h = silu(gate) * up, rounded to bf16 in bf16 mode (the dtype the down
    GEMM consumes), y[t] = sum over the token's k slots, in slot order, of
    route_w * (h @ W_down^T).

  * MoE routing (a DeepSeekV3/Kimi-style MoE whose routing includes a shared
    expert: [QC] "The Context: A Native DDTree Engine Takes Shape" and [PC]
    "The Context: Phase 3 of a Custom Inference Stack"; the pages give no
    formula, so the published DeepSeek-V3 gate is taken): fp32 router
    logits l = x @ W_r^T, scores s = sigmoid(l), the k experts with the
    largest s + b (b an optional per-expert selection bias; equal values go
    to the lower expert id), weights s_j / sum of the k chosen s times a
    routing scale;
  * shared expert: a SwiGLU expert that every token uses with weight 1,
    added after the routed slots.

Every function is pinned by tests against closed forms, brute force and
invariants (tests/test_oracle_pins.py); none is "parity unpinned".
"""

from __future__ import annotations

import numpy as np

GROUP = 32          # [QC] "Input Knowledge Required": group size 32
NIB_PER_WORD = 8    # [QC] "The INT4 Milestone": 8 nibbles per int32
ZERO_POINT = 8      # [QC] "Input Knowledge Required": value = nibble - 8
QMAX = 7            # symmetric range: max|w| maps to 7


# --------------------------------------------------------------- format
def pack_nibbles(nib: np.ndarray) -> np.ndarray:
    """nib[N, K] in 0..15 -> qw[N, K/8] int32, nibble k%8 in bits 4*(k%8).

    [QC] "The INT4 Milestone": 8 nibbles per int32 along the input dim.
    """
    nib = np.asarray(nib)
    N, K = nib.shape
    if K % NIB_PER_WORD:
        raise ValueError("K must be a multiple of 8")
    if nib.min(initial=0) < 0 or nib.max(initial=0) > 15:
        raise ValueError("nibbles must be in 0..15")
    n = nib.astype(np.uint32).reshape(N, K // NIB_PER_WORD, NIB_PER_WORD)
    word = np.zeros((N, K // NIB_PER_WORD), dtype=np.uint32)
    for j in range(NIB_PER_WORD):
        word |= n[:, :, j] << np.uint32(4 * j)
    return word.view(np.int32)


def unpack_nibbles(qw: np.ndarray) -> np.ndarray:
    """qw[N, K/8] int32 -> nib[N, K] uint8 (logical shifts of the bit pattern)."""
    u = np.ascontiguousarray(qw).view(np.uint32)
    N, W = u.shape
    nib = np.empty((N, W, NIB_PER_WORD), dtype=np.uint8)
    for j in range(NIB_PER_WORD):
        nib[:, :, j] = (u >> np.uint32(4 * j)) & np.uint32(0xF)
    return nib.reshape(N, W * NIB_PER_WORD)


def quantize_w4a16(w: np.ndarray, group: int = GROUP):
    """Symmetric per-group INT4 quantiser: w[N, K] fp32 -> (qw, sc).

    [QC] "The INT4 Milestone" (quantize_w4a16, symmetric, nibble = q + 8).
    For each row and each group of ``group`` consecutive k:
        s = max|w| / 7                     (fp32)
        q = clamp(round_half_even(w / s), -8, 7)   (fp32 division; q = 0 if s = 0)
        nibble = q + 8
    Returns qw[N, K/8] int32 and sc[N, K/group] fp32.
    """
    w = np.ascontiguousarray(w, dtype=np.float32)
    N, K = w.shape
    if K % group:
        raise ValueError("K must be a multiple of the group size")
    G = K // group
    wg = w.reshape(N, G, group)
    s = (np.abs(wg).max(axis=2) / np.float32(QMAX)).astype(np.float32)      # [N, G]
    safe = np.where(s > 0, s, np.float32(1.0)).astype(np.float32)
    ratio = (wg / safe[:, :, None]).astype(np.float32)                      # fp32 division
    q = np.rint(ratio)                                                      # half to even
    q = np.where(s[:, :, None] > 0, q, 0.0)
    q = np.clip(q, -ZERO_POINT, QMAX).astype(np.int64)
    nib = (q + ZERO_POINT).reshape(N, K)
    return pack_nibbles(nib), s


def dequantize(qw: np.ndarray, sc: np.ndarray, group: int = GROUP) -> np.ndarray:
    """W_hat[N, K] fp32 = (nibble - 8) * scale, as an fp32 product.

    [QC] "The INT4 Milestone" / "Input Knowledge Required" (value = nibble - 8).
    """
    nib = unpack_nibbles(qw)
    N, K = nib.shape
    sc = np.asarray(sc, dtype=np.float32)
    if sc.shape != (N, K // group):
        raise ValueError("scale shape mismatch")
    q = (nib.astype(np.int32) - ZERO_POINT).astype(np.float32)
    return (q * np.repeat(sc, group, axis=1)).astype(np.float32)


def round_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to the nearest bf16 (ties to even); returned as fp32."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)) << np.uint64(16)
    out = (r & np.uint64(0xFFFFFFFF)).astype(np.uint32).view(np.float32)
    nan = np.isnan(a)
    if nan.any():
        out = out.copy()
        out[nan] = np.float32(np.nan)
    return out


# --------------------------------------------------------------- GEMM
def gemm_ref(x: np.ndarray, qw: np.ndarray, sc: np.ndarray, group: int = GROUP):
    """y[M, N] = sum_k x[m, k] * W_hat[n, k], accumulated in fp64.

    [SoS] "The Weight of Context" (dequantise-then-multiply golden);
    [QC] "The INT4 Milestone" (fp32 activations x int4 weights + scales).
    ``x`` is fp32, or the bf16 values of a bf16 activation (as fp32).
    Returns (y, bound) where bound[m, n] = sum_k |x[m, k] * W_hat[n, k]|,
    the scale that the error tolerances are stated against.
    """
    x64 = np.asarray(x, dtype=np.float32).astype(np.float64)
    w64 = dequantize(qw, sc, group).astype(np.float64)
    if x64.shape[1] != w64.shape[1]:
        raise ValueError("K mismatch")
    y = x64 @ w64.T
    bound = np.abs(x64) @ np.abs(w64).T
    return y, bound


# --------------------------------------------------------------- MoE
def silu(g: np.ndarray) -> np.ndarray:
    """silu(g) = g / (1 + exp(-g)), fp64."""
    g = np.asarray(g, dtype=np.float64)
    return g / (1.0 + np.exp(-g))


def moe_sort(expert_ids: np.ndarray, E: int):
    """Group (token, slot) pairs by expert, stably.

    Pair p = t * topk + slot. offsets[e] = number of pairs with expert < e
    (exclusive prefix sum of the histogram, offsets[E] = T * topk) and perm
    lists the pairs ordered by (expert, p) ascending.
    """
    ids = np.asarray(expert_ids, dtype=np.int64).reshape(-1)
    if ids.size and (ids.min() < 0 or ids.max() >= E):
        raise ValueError("expert id out of range")
    counts = np.bincount(ids, minlength=E)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    perm = np.argsort(ids, kind="stable")
    return offsets.astype(np.int32), perm.astype(np.int32)


def _silu_slope_max() -> float:
    # max over g of d/dg silu(g) is about 1.0998; 1.1 bounds it.
    return 1.1


def _swiglu_one(wgu, xt, eps, slope):
    """Exact SwiGLU of one token through one expert (wgu dequantised, fp64)
    and the bound dh on |h_impl - h| for an implementation whose gate/up GEMM
    stays within eps * sum|x * w| and which evaluates silu and the product in
    fp32 (first-order propagation through SwiGLU)."""
    I = wgu.shape[0] // 2
    gu = wgu @ xt
    bgu = np.abs(wgu) @ np.abs(xt)
    g, u = gu[:I], gu[I:]
    dg, du = eps * bgu[:I], eps * bgu[I:]
    h = silu(g) * u
    dh = slope * (np.abs(u) + du) * dg + np.abs(silu(g)) * du + 4e-7 * np.abs(h)
    return h, dh


def moe_swiglu_ref(x, qw_gu, sc_gu, bf16_mode: bool, eps: float, group: int = GROUP):
    """The gate/up GEMM and SwiGLU of ONE expert for tokens x[m, H].

    [QC] "The Context: A Native DDTree Engine Takes Shape" (SwiGLU between
    the expert GEMMs): [g; u] = x @ W_hat_gu^T, h = silu(g) * u.
    Returns (h, tol): h [m, I] exact in fp64, and tol [m, I] such that an
    implementation whose gate/up GEMM stays within eps * sum|x * w|, which
    evaluates silu and the product in fp32 and, in bf16 mode, stores h
    rounded to bf16 (nearest, 2^-9 relative), is within tol of h.
    """
    x = np.asarray(x, dtype=np.float32)
    wgu = dequantize(qw_gu, sc_gu, group).astype(np.float64)
    I = wgu.shape[0] // 2
    h = np.zeros((x.shape[0], I))
    tol = np.zeros((x.shape[0], I))
    for m in range(x.shape[0]):
        h[m], dh = _swiglu_one(wgu, x[m].astype(np.float64), eps, _silu_slope_max())
        tol[m] = dh * (1 + 2.0 ** -9) + 2.0 ** -9 * np.abs(h[m]) if bf16_mode else dh
    return h, tol


def moe_down_ref(h_in, route_w, qw_dn, sc_dn, eps: float, group: int = GROUP):
    """The down GEMM of ONE expert fed the given h, times the routing weight.

    [QC] "The Context: A Native DDTree Engine Takes Shape" (the down
    projection after SwiGLU); the routing weight scales each slot's output.
    o[m] = route_w[m] * (h_in[m] @ W_hat_dn^T), exact in fp64. Returns
    (o, tol): tol = |route_w| * eps * (|h_in| @ |W_hat_dn|^T) (a GEMM within
    eps of sum|h * w|) plus 2^-23 |o| (the fp32 product by the routing
    weight and its rounding).
    """
    h_in = np.asarray(h_in, dtype=np.float64)
    r = np.asarray(route_w, dtype=np.float32).astype(np.float64)
    wdn = dequantize(qw_dn, sc_dn, group).astype(np.float64)
    o = r[:, None] * (h_in @ wdn.T)
    tol = np.abs(r)[:, None] * eps * (np.abs(h_in) @ np.abs(wdn).T) + 2.0 ** -23 * np.abs(o)
    return o, tol


def moe_ref(x, expert_ids, route_w, qw_gu, sc_gu, qw_dn, sc_dn, bf16_mode: bool,
            eps: float, group: int = GROUP, tokens=None):
    """Grouped MoE layer: y[t] = sum_slot r[t,slot] * (h @ W_dn[e]^T).

    [QC] "The Context: A Native DDTree Engine Takes Shape" (MoE with SwiGLU),
    "The INT4 Milestone" (experts run through the INT4 path);
    [PC] "The Context: Phase 3 ..." (INT4 W4A16 group-quantised MoE path).
    For token t and slot j with expert e = expert_ids[t, j]:
        [g; u] = x[t] @ W_hat_gu[e]^T   (g = rows 0..I-1, u = rows I..2I-1)
        h      = silu(g) * u            (rounded to bf16 in bf16 mode)
        o      = route_w[t, j] * (h @ W_hat_dn[e]^T)
        y[t]   = o[slot 0] + o[slot 1] + ... in slot order.
    ``qw_gu``/``sc_gu``/``qw_dn``/``sc_dn`` are indexable by expert id
    (arrays [E, ...] or a mapping). ``tokens`` optionally restricts the
    computation to a list of token indices (rows of the result); the others
    are left at zero.

    Returns (y, tol): tol[t, n] is a per-output error bound for an
    implementation whose two GEMMs each stay within eps * sum|a * w| of the
    exact product, derived by propagating those bounds through SwiGLU, the
    bf16 rounding of h, the routing weight and the slot sum.
    """
    x = np.asarray(x, dtype=np.float32)
    T, H = x.shape
    ids = np.asarray(expert_ids)
    topk = ids.shape[1]
    r = np.asarray(route_w, dtype=np.float32).astype(np.float64)
    toks = np.arange(T) if tokens is None else np.asarray(sorted(set(int(t) for t in tokens)))
    o = {}      # (t, slot) -> (o, bound on |o - o_exact|, |o|)
    slope = _silu_slope_max()
    by_expert = {}
    for t in toks:
        for j in range(topk):
            by_expert.setdefault(int(ids[t, j]), []).append((int(t), j))
    for e in sorted(by_expert):
        wgu = dequantize(qw_gu[e], sc_gu[e], group).astype(np.float64)
        wdn = dequantize(qw_dn[e], sc_dn[e], group).astype(np.float64)
        for (t, j) in by_expert[e]:
            h, dh = _swiglu_one(wgu, x[t].astype(np.float64), eps, slope)
            if bf16_mode:
                h_in = round_to_bf16(h.astype(np.float32)).astype(np.float64)
                # both sides round h to bf16: a rounding flip costs up to one
                # bf16 ulp of the operand (2^-8 relative)
                dh = dh * (1 + 2.0 ** -9) + 2.0 ** -8 * np.abs(h_in)
            else:
                h_in = h
            oo = r[t, j] * (wdn @ h_in)
            do = abs(r[t, j]) * (eps * (np.abs(wdn) @ np.abs(h_in)) + np.abs(wdn) @ dh)
            o[(t, j)] = (oo, do, np.abs(oo))
    y = np.zeros((T, H), dtype=np.float64)
    tol = np.zeros((T, H), dtype=np.float64)
    for t in toks:
        absacc = np.zeros(H, dtype=np.float64)
        for j in range(topk):           # slot order
            oo, do, ao = o[(int(t), j)]
            y[t] += oo
            tol[t] += do
            absacc += ao
        # the fp32 routing-weight product and the fp32 slot sum
        tol[t] += (topk + 2) * 2.0 ** -24 * absacc
    return y, tol


def sigmoid(v: np.ndarray) -> np.ndarray:
    """Logistic function 1 / (1 + exp(-v)) in fp64."""
    v = np.asarray(v, dtype=np.float64)
    return 1.0 / (1.0 + np.exp(-v))


def moe_route_ref(x, router_w, bias, topk: int, route_scale: float):
    """Router of the MoE block: logits, top-k expert ids and routing weights.

    [QC] "The Context: A Native DDTree Engine Takes Shape" and [PC] "The
    Context: Phase 3 of a Custom Inference Stack" (DeepSeekV3/Kimi-style MoE
    routing); the gate itself is the published DeepSeek-V3 one:
        l[t, e]  = x[t] . W_r[e]                      (x as given, fp32 values)
        s[t, e]  = sigmoid(l[t, e])
        ids[t]   = the topk experts with the largest s + b, in decreasing
                   order of s + b; equal values go to the lower expert id
        w[t, j]  = route_scale * s[t, ids[t, j]] / sum_j' s[t, ids[t, j']]
    ``bias`` may be None (all zero). Returns (logits, bound, ids, w):
    logits and bound = |x| @ |W_r|^T in fp64, ids int32 [T, topk], w fp64.
    """
    x64 = np.asarray(x, dtype=np.float32).astype(np.float64)
    wr = np.asarray(router_w, dtype=np.float32).astype(np.float64)
    T = x64.shape[0]
    E = wr.shape[0]
    if not 1 <= topk <= E:
        raise ValueError("topk must be in 1..E")
    logits = x64 @ wr.T
    bound = np.abs(x64) @ np.abs(wr).T
    s = sigmoid(logits)
    b = np.zeros(E) if bias is None else np.asarray(bias, dtype=np.float32).astype(np.float64)
    sel = s + b
    ids = np.zeros((T, topk), dtype=np.int32)
    w = np.zeros((T, topk), dtype=np.float64)
    for t in range(T):
        # a stable sort on -sel keeps equal values in increasing expert id
        order = np.argsort(-sel[t], kind="stable")[:topk]
        ids[t] = order
        w[t] = route_scale * s[t, order] / np.sum(s[t, order])
    return logits, bound, ids, w


class _ExpertsWithShared:
    """Expert tensors indexable by id: the routed ones, then the shared one at id E."""

    def __init__(self, routed, shared, E):
        self.routed, self.shared, self.E = routed, shared, E

    def __getitem__(self, e):
        return self.shared if e == self.E else self.routed[e]


def moe_block_ref(x, expert_ids, route_w, qw_gu, sc_gu, qw_dn, sc_dn, shared, bf16_mode: bool,
                  eps: float, group: int = GROUP, tokens=None):
    """MoE block: the routed layer of ``moe_ref`` plus the shared expert.

    [QC] "The Context: A Native DDTree Engine Takes Shape" and "The INT4
    Milestone" (MoE routing with a shared expert; routed and shared experts
    run through the INT4 path). ``shared`` is (qw_gu_s, sc_gu_s, qw_dn_s,
    sc_dn_s) of one SwiGLU expert (its width may differ from the routed
    experts'), or None. The shared expert is an extra slot after the routed
    ones, used by every token with weight 1:
        y[t] = sum_j w[t, j] * expert_{ids[t, j]}(x[t]) + expert_shared(x[t]).
    Returns (y, tol) as ``moe_ref``.
    """
    if shared is None:
        return moe_ref(x, expert_ids, route_w, qw_gu, sc_gu, qw_dn, sc_dn, bf16_mode, eps,
                       group, tokens)
    ids = np.asarray(expert_ids)
    T, topk = ids.shape
    E = len(qw_gu) if not isinstance(qw_gu, dict) else max(qw_gu) + 1
    E = max(E, int(ids.max()) + 1)
    ids_ext = np.concatenate([ids, np.full((T, 1), E, dtype=ids.dtype)], axis=1)
    w_ext = np.concatenate([np.asarray(route_w, dtype=np.float64), np.ones((T, 1))], axis=1)
    m = [_ExpertsWithShared(a, b, E) for a, b in zip((qw_gu, sc_gu, qw_dn, sc_dn), shared)]
    return moe_ref(x, ids_ext, w_ext, m[0], m[1], m[2], m[3], bf16_mode, eps, group, tokens)
