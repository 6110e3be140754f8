"""Seeded synthetic inputs for the W4A16 group-GEMM workloads.

This module only draws random numbers. It holds none of the method's
arithmetic (no quantisation, packing, dequantisation or products), so both
the CPU oracle and the CUDA path can take their inputs from it without
sharing any of the computation under test.

Recipes (all seeded, no dataset):
  * activations  x ~ N(0, 1) fp32; optionally a fixed fraction of entries,
    chosen by seeded sampling without replacement, multiplied by an outlier
    factor (the tree-verify workload uses 1 % of entries x20);
  * weights      W ~ N(0, 1/K) fp32 (std 1/sqrt(K)), one matrix per call;
  * MoE routing  per token, top-k distinct experts drawn uniformly without
    replacement, and routing weights that are the softmax of k N(0,1)
    logits (the routing weights are an input of the grouped GEMM, not
    something it computes).

Host draws use numpy's PCG64 keyed by (seed, stream); device draws (for the
workloads too large to synthesise on the host in reasonable time) use
torch's CUDA generator keyed by a seed derived from the same pair. The two
families are different streams; a test that needs the same values on both
sides copies the drawn tensor, it never redraws it on the other side.
"""

from __future__ import annotations

import numpy as np

# Stream identifiers keep unrelated draws independent for one seed.
STREAM_X = 1
STREAM_W = 2
STREAM_OUTLIER = 3
STREAM_ROUTE_IDS = 4
STREAM_ROUTE_LOGITS = 5


def _rng(seed: int, stream: int, sub: int = 0) -> np.random.Generator:
    return np.random.default_rng([int(seed), int(stream), int(sub)])


def activations(seed: int, M: int, K: int, outlier_frac: float = 0.0,
                outlier_scale: float = 20.0, sub: int = 0) -> np.ndarray:
    """x[M, K] fp32 ~ N(0,1); floor(outlier_frac*M*K) distinct entries scaled."""
    x = _rng(seed, STREAM_X, sub).standard_normal((M, K), dtype=np.float32)
    n_out = int(np.floor(outlier_frac * M * K))
    if n_out > 0:
        pos = _rng(seed, STREAM_OUTLIER, sub).choice(M * K, size=n_out, replace=False)
        flat = x.reshape(-1)
        flat[pos] = flat[pos] * np.float32(outlier_scale)
    return x


def weights(seed: int, N: int, K: int, sub: int = 0) -> np.ndarray:
    """W[N, K] fp32 ~ N(0, 1/K)."""
    w = _rng(seed, STREAM_W, sub).standard_normal((N, K), dtype=np.float32)
    return w * np.float32(1.0 / np.sqrt(K))


def routing(seed: int, T: int, topk: int, E: int):
    """Expert ids [T, topk] int32 (distinct per token) and weights [T, topk] fp32.

    Ids: a partial Fisher-Yates shuffle of range(E) per token (uniform, without
    replacement). Weights: softmax over the token's topk N(0,1) logits,
    evaluated in fp64 and stored as fp32.
    """
    if topk > E:
        raise ValueError("topk > E")
    rng = _rng(seed, STREAM_ROUTE_IDS)
    ids = np.empty((T, topk), dtype=np.int32)
    for t in range(T):
        perm = np.arange(E)
        for i in range(topk):
            j = int(rng.integers(i, E))
            perm[i], perm[j] = perm[j], perm[i]
        ids[t] = perm[:topk]
    logits = _rng(seed, STREAM_ROUTE_LOGITS).standard_normal((T, topk))
    z = np.exp(logits - logits.max(axis=1, keepdims=True))
    w = (z / z.sum(axis=1, keepdims=True)).astype(np.float32)
    return ids, w


# ---------------------------------------------------------------- device side
def _device_seed(seed: int, stream: int, sub: int) -> int:
    ss = np.random.SeedSequence([int(seed), int(stream), int(sub), 0xD5])
    return int(ss.generate_state(1, dtype=np.uint64)[0] & ((1 << 63) - 1))


def weights_device(seed: int, N: int, K: int, device, sub: int = 0):
    """W[N, K] fp32 ~ N(0, 1/K) drawn on the device (torch CUDA generator)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(_device_seed(seed, STREAM_W, sub))
    w = torch.randn((N, K), generator=g, device=device, dtype=torch.float32)
    w.mul_(float(1.0 / np.sqrt(K)))
    return w


def activations_device(seed: int, M: int, K: int, device, sub: int = 0):
    """x[M, K] fp32 ~ N(0, 1) drawn on the device (torch CUDA generator)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(_device_seed(seed, STREAM_X, sub))
    return torch.randn((M, K), generator=g, device=device, dtype=torch.float32)
