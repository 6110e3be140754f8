"""Benchmark of the W4A16 group-quantised GEMM library on one GB300.

Headline workload (the JSON line's `value`): the decode GEMV, M=1, K=7168,
N=4096 (fused gate+up of an MoE expert), group 32, fp32 activations. A step
is one w4a16_gemm call; the metric is effective TB/s = algorithmic bytes
(packed weights + scales + activations + output) / time.

Every other workload is measured in the same run, with the same steps,
warm-up and L2 policy, and reported under `configs`:
  0      tiny GEMM 1x256 -> 512 fp32             (TB/s; launch-latency bound)
  2-f32  tree-verify pair M=64 (7168->4096 then 2048->7168), fp32 activations
  2-bf16 the same pair, bf16 activations          (TB/s)
  3      grouped MoE layer: 128 tokens, 384 experts, top-8, bf16 (TB/s of
         active-expert bytes)
  4      prefill GEMM 2048x7168 -> 18432 bf16     (TFLOP/s)
  5      whole MoE block: layer 3 plus the router and one shared expert
         (width 2048), bf16                       (TB/s of active bytes)
`--config KEY` makes another workload the headline; `--only` skips the rest.

Timing: W eager warm-up steps, then exactly K steps captured in one CUDA
graph and replayed once between barrier + synchronize, timed with CUDA
events on the launching stream; max over ranks. Before the start event the
stream is kept busy by a spin kernel, so that the time the host takes to
enqueue the graph is not counted as device time; two more spin kernels of a
known cycle count, timed with their own events just before and just after
the timed region, give the SM clock of that moment. Working sets below the
L2 size rotate through enough weight copies that every step reads its
weights from HBM. `e2e` repeats the steps through the Python binding with
the per-step inputs copied in from pinned host memory and the result copied
back and waited for.

Oracle legs (CPU baseline, `--impl reference`): the oracle (numpy fp64) on a
bounded sample of the same workload, with weights quantised by the oracle's
own quantiser on the host from the same seeded draws; those legs never
import the CUDA library.

Multi-GPU: independent replicas (the path is not partitioned across GPUs);
value = all ranks' bytes / max time, scaling "weak".
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
METRIC = "w4a16_gemm effective TB/s (small M) & TFLOP/s (large M), % of GB300 roofline"
L2_BYTES = 129 * 2 ** 20
ALL_CONFIGS = ["0", "1", "2-f32", "2-bf16", "3", "4", "5"]
# Spin-kernel lengths (SM clock cycles): the hold before the timed region
# and the two clock probes around it.
HOLD_CYCLES = 2_000_000
CLOCK_PROBE_CYCLES = 400_000


# ----------------------------------------------------------------- helpers
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
            "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "int4_w4a16_group_gemm_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_key):
    """DRAM bytes per launch from a committed ncu summary, if current."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    cur = kernel_source_hash()
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 3 and not line.startswith("#") and parts[0] == kernel_key:
                return float(parts[1]) if parts[2] == cur else None
    return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the GPU works."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0):
        self.index = index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()
        time.sleep(0.2)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        return summarise_clock_lines([ln for _, ln in self.lines])


def summarise_clock_lines(lines):
    """Median SM clock of the busy samples, max clock, active slowdown reasons."""
    sm, smax, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for ln in lines:
        f = [v.strip() for v in ln.split(",")]
        if len(f) < 9:
            continue
        try:
            sm.append(float(f[1]))
            smax.append(float(f[2]))
        except ValueError:
            continue
        for n, v in zip(names, f[5:9]):
            if v.lower().startswith("active"):
                reasons.add(n)
    if not sm:
        return None
    busy = [s for s in sm if s > 0.5 * max(sm)] or sm
    return {"sm_mhz": float(np.median(busy)), "sm_max_mhz": float(max(smax)),
            "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------- workload specs
def _gemm_bytes(M, N, K, xbytes, group=32):
    return N * K // 2 + N * (K // group) * 4 + M * K * xbytes + M * N * 4


def _rotation(bytes_per_copy):
    return max(1, int(np.ceil(4.0 * L2_BYTES / bytes_per_copy)))


MOE_T, MOE_H, MOE_I, MOE_E, MOE_TOPK, SHARED_I = 128, 7168, 2048, 384, 8, 2048

GEMM_SPECS = {
    # key: (M, N, K, dtype, seed, outlier, name)
    "0": (1, 512, 256, "f32", 0, 0.0, "tiny GEMM M=1 K=256 N=512 group=32 fp32 activations"),
    "1": (1, 4096, 7168, "f32", 0, 0.0,
          "decode GEMV M=1 K=7168 N=4096 group=32 fp32 activations"),
    "4": (2048, 18432, 7168, "bf16", 0, 0.0,
          "prefill GEMM M=2048 K=7168 N=18432 group=32 bf16 activations"),
}
PAIR_SPEC = [(64, 4096, 7168, 0, "a"), (64, 7168, 2048, 1, "b")]  # M, N, K, seed, tag


def workload_config(key, moe_experts=MOE_E, moe_tokens=MOE_T):
    """The `config` object of a workload: identical in both arms."""
    if key in GEMM_SPECS:
        M, N, K, dt, _, _, name = GEMM_SPECS[key]
        wbytes = N * K // 2 + N * (K // 32) * 4
        l2 = (f"{_rotation(wbytes)} rotating weight copies (> 4x L2)" if wbytes < 2 * L2_BYTES
              else "working set larger than L2")
        return {"workload": name, "config_index": key, "M": M, "N": N, "K": K, "group": 32,
                "activations": dt, "l2": l2}
    if key in ("2-f32", "2-bf16"):
        dt = key.split("-")[1]
        rot = [_rotation(N * K // 2 + N * (K // 32) * 4) for _, N, K, _, _ in PAIR_SPEC]
        return {"workload": f"tree-verify pair M=64 (7168->4096, 2048->7168) group=32 {dt}",
                "config_index": key, "M": 64, "shapes": "4096x7168, 7168x2048",
                "activations": dt, "outliers": "1% of entries x20",
                "l2": f"{rot[0]} / {rot[1]} rotating weight copies (> 4x L2)"}
    if key == "3":
        return {"workload": (f"grouped MoE T={moe_tokens} H={MOE_H} I={MOE_I} E={moe_experts} "
                             f"top-{MOE_TOPK} group=32 bf16"),
                "config_index": key, "activations": "bf16",
                "routing": "uniform top-8 without replacement, softmax(N(0,1)) weights",
                "l2": "working set larger than L2"}
    if key == "5":
        return {"workload": (f"MoE block T={moe_tokens} H={MOE_H} I={MOE_I} E={moe_experts} "
                             f"top-{MOE_TOPK} + shared expert Is={SHARED_I}, router fp32, bf16"),
                "config_index": key, "activations": "bf16",
                "routing": "device router: sigmoid top-8 with bias 0.05 N(0,1), scale 2.827",
                "l2": "working set larger than L2"}
    raise ValueError(key)


# ----------------------------------------------------------------- host inputs (both arms)
def _bf16_round(x):
    import torch
    return torch.from_numpy(x).to(torch.bfloat16).float().numpy()


def gemm_host_inputs(M, N, K, dt, seed, outlier):
    """x (fp32 values; bf16-representable in bf16 mode) and W, seeded, on the host."""
    import synth
    x = synth.activations(seed, M, K, outlier_frac=outlier)
    if dt == "bf16":
        x = _bf16_round(x)
    return x, synth.weights(seed, N, K)


def oracle_gemm_sample(x, w, budget_s, group=32):
    """Time oracle.gemm_ref on a row sample of W (quantised by the oracle's own
    quantiser, outside the timing); -> (seconds per full call, description)."""
    import oracle
    N = w.shape[0]
    q64, s64 = oracle.quantize_w4a16(w[:min(64, N)], group)
    t0 = time.perf_counter()
    oracle.gemm_ref(x, q64, s64, group)
    per_row = (time.perf_counter() - t0) / q64.shape[0]
    rows = int(max(min(N, 8), min(N, budget_s / 3 / max(per_row, 1e-9))))
    qw, sc = oracle.quantize_w4a16(w[:rows], group)
    reps = 0
    t0 = time.perf_counter()
    while True:
        oracle.gemm_ref(x, qw, sc, group)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= 50:
            break
    per_call = el / reps * N / rows
    return per_call, (f"{reps} x oracle.gemm_ref on {rows} of {N} weight rows (M={x.shape[0]}), "
                      f"scaled to the full call")


def moe_host_experts(experts, seed, dev):
    """Oracle-quantised weights of the given experts, from the same device
    draws the GPU arm quantises (copied to the host; input synthesis only)."""
    import oracle
    import synth
    out = {}
    for e in experts:
        wgu = synth.weights_device(seed, 2 * MOE_I, MOE_H, dev, sub=2 * e).cpu().numpy()
        wdn = synth.weights_device(seed, MOE_H, MOE_I, dev, sub=2 * e + 1).cpu().numpy()
        out[e] = oracle.quantize_w4a16(wgu) + oracle.quantize_w4a16(wdn)
    return out


def oracle_moe_sample(x, ids, rw, experts, tokens, shared=None, router=None):
    """Time the oracle's MoE layer (or block) on `tokens`; -> (seconds per
    full call, description). `experts` maps id -> (qw_gu, sc_gu, qw_dn, sc_dn)."""
    import oracle
    T = x.shape[0]
    m = [{e: v[i] for e, v in experts.items()} for i in range(4)]
    t0 = time.perf_counter()
    if router is not None:
        wr, bias, topk, scale = router
        oracle.moe_route_ref(x[tokens], wr, bias, topk, scale)
    if shared is None:
        oracle.moe_ref(x, ids, rw, *m, True, eps=4e-3, tokens=tokens)
    else:
        oracle.moe_block_ref(x, ids, rw, *m, shared, True, eps=4e-3, tokens=tokens)
    el = time.perf_counter() - t0
    what = "router + moe_block_ref" if shared is not None else "moe_ref"
    return el / len(tokens) * T, (f"oracle {what} on {len(tokens)} of {T} tokens "
                                  f"({len(experts)} experts), scaled by tokens")


# ----------------------------------------------------------------- GPU workloads
class Workload:
    """One configuration: device buffers, a step, its bytes and flops."""

    key = ""
    unit = "TB/s"
    dtype = "f32"
    bound = "hbm"
    kernels_per_step = 1

    def step(self, i, stream):
        raise NotImplementedError

    def e2e_step(self, i, stream):
        raise NotImplementedError

    def oracle_sample(self, budget_s):
        raise NotImplementedError

    def rate(self, seconds):
        return (self.flops if self.unit == "TFLOP/s" else self.bytes) / seconds / 1e12


class GemmWorkload(Workload):
    def __init__(self, w4, torch, dev, M, N, K, dtype, seed, outlier=0.0, algo="auto",
                 overlap=True, name=""):
        self.w4, self.torch, self.dev = w4, torch, dev
        self.M, self.N, self.K = M, N, K
        self.dtype = dtype
        self.name = name
        self.algo = algo
        self.overlap = overlap
        wbytes = N * K // 2 + N * (K // 32) * 4
        self.bytes = _gemm_bytes(M, N, K, 2 if dtype == "bf16" else 4)
        self.flops = 2.0 * M * N * K
        self.ncopies = _rotation(wbytes) if wbytes < 2 * L2_BYTES else 1
        self.x_np, self.w_np = gemm_host_inputs(M, N, K, dtype, seed, outlier)
        wd = torch.from_numpy(self.w_np).to(dev)
        self.qw, self.sc = [], []
        for _ in range(self.ncopies):
            qw, sc = w4.w4a16_quantize(wd)
            self.qw.append(qw)
            self.sc.append(sc)
        del wd
        xt = torch.from_numpy(self.x_np)
        if dtype == "bf16":
            xt = xt.to(torch.bfloat16)
        self.x_host = xt.pin_memory()
        self.x = self.x_host.to(dev)
        self.y = torch.empty((M, N), dtype=torch.float32, device=dev)
        self.y_host = torch.empty((M, N), dtype=torch.float32).pin_memory()
        self.h2d = self.x_host.numel() * self.x_host.element_size()
        self.d2h = self.y_host.numel() * 4
        if M >= 1024:
            self.unit, self.bound = "TFLOP/s", "tensor"
        n = w4.w4a16_gemm_launches(M, N, K, dtype, algo)
        if n <= 0:
            raise RuntimeError(f"gemm rejected: status {-n}")
        self.kernels_per_step = n

    def step(self, i, stream):
        c = i % self.ncopies
        self.w4.w4a16_gemm(self.x, self.qw[c], self.sc[c], y=self.y, algo=self.algo,
                           overlap=self.overlap, stream=stream)

    def e2e_step(self, i, stream):
        c = i % self.ncopies
        self.x.copy_(self.x_host, non_blocking=True)
        self.w4.w4a16_gemm(self.x, self.qw[c], self.sc[c], y=self.y, algo=self.algo,
                           overlap=self.overlap, stream=stream)
        self.y_host.copy_(self.y, non_blocking=True)
        stream.synchronize()

    def oracle_sample(self, budget_s):
        per_call, desc = oracle_gemm_sample(self.x_np, self.w_np, budget_s)
        return self.rate(per_call), desc


class PairWorkload(Workload):
    """The two M=64 GEMMs of a tree-verify step (7168->4096, 2048->7168)."""

    def __init__(self, w4, torch, dev, dtype, overlap=True):
        self.parts = [GemmWorkload(w4, torch, dev, M, N, K, dtype, seed, outlier=0.01,
                                   overlap=overlap, name=tag)
                      for M, N, K, seed, tag in PAIR_SPEC]
        self.name = f"tree-verify pair M=64 {dtype}"
        self.dtype = dtype
        self.bytes = sum(p.bytes for p in self.parts)
        self.flops = sum(p.flops for p in self.parts)
        self.h2d = sum(p.h2d for p in self.parts)
        self.d2h = sum(p.d2h for p in self.parts)
        self.kernels_per_step = sum(p.kernels_per_step for p in self.parts)
        # bf16: HBM-bound on the tensor cores. fp32: the fp32-exact tensor-core
        # kernel multiplies three bf16 pieces of every activation, so its
        # tensor work is 3 x 2MNK, which outweighs the HBM time at M = 64.
        self.bound = "hbm" if dtype == "bf16" else "tensor"
        self.tensor_factor = 1.0 if dtype == "bf16" else 3.0

    def step(self, i, stream):
        for p in self.parts:
            p.step(i, stream)

    def e2e_step(self, i, stream):
        for p in self.parts:
            p.e2e_step(i, stream)

    def oracle_sample(self, budget_s):
        ta, da = oracle_gemm_sample(self.parts[0].x_np, self.parts[0].w_np, budget_s / 2)
        tb, db = oracle_gemm_sample(self.parts[1].x_np, self.parts[1].w_np, budget_s / 2)
        return self.bytes / (ta + tb) / 1e12, f"{da}; {db}"


class MoeWorkload(Workload):
    """Grouped MoE layer: 128 tokens, hidden 7168, 384 experts (I=2048), top-8, bf16."""

    def __init__(self, w4, torch, dev, seed=0, T=MOE_T, E=MOE_E):
        import synth
        H, I, topk = MOE_H, MOE_I, MOE_TOPK
        self.w4, self.torch, self.dev, self.seed = w4, torch, dev, seed
        self.T, self.H, self.I, self.E, self.topk = T, H, I, E, topk
        self.name = f"grouped MoE T={T} H={H} I={I} E={E} top-{topk} bf16"
        self.dtype = "bf16"
        self.qgu = torch.empty((E, 2 * I, H // 8), dtype=torch.int32, device=dev)
        self.sgu = torch.empty((E, 2 * I, H // 32), dtype=torch.float32, device=dev)
        self.qdn = torch.empty((E, H, I // 8), dtype=torch.int32, device=dev)
        self.sdn = torch.empty((E, H, I // 32), dtype=torch.float32, device=dev)
        for e in range(E):
            w4.w4a16_quantize(synth.weights_device(seed, 2 * I, H, dev, sub=2 * e),
                              qw=self.qgu[e], sc=self.sgu[e])
            w4.w4a16_quantize(synth.weights_device(seed, H, I, dev, sub=2 * e + 1),
                              qw=self.qdn[e], sc=self.sdn[e])
        self.x_np = _bf16_round(synth.activations(seed, T, H))
        ids, rw = synth.routing(seed, T, topk, E)
        self.ids_np, self.rw_np = ids, rw
        self.x_host = torch.from_numpy(self.x_np).to(torch.bfloat16).pin_memory()
        self.ids_host = torch.from_numpy(ids).pin_memory()
        self.rw_host = torch.from_numpy(rw).pin_memory()
        self.x = self.x_host.to(dev)
        self.ids = self.ids_host.to(dev)
        self.rw = self.rw_host.to(dev)
        self.ws = torch.empty(w4.w4a16_moe_workspace_size(T, topk, E, H, I), dtype=torch.uint8,
                              device=dev)
        self.y = torch.empty((T, H), dtype=torch.float32, device=dev)
        self.y_host = torch.empty((T, H), dtype=torch.float32).pin_memory()
        self.active = len(set(int(e) for e in ids.reshape(-1)))
        self.per_expert = (2 * I * H // 2 + 2 * I * (H // 32) * 4) + (H * I // 2 + H * (I // 32) * 4)
        self.bytes = self.active * self.per_expert + T * H * 2 + T * H * 4
        self.flops = 2.0 * T * topk * (2 * I * H + H * I)
        self.h2d = (self.x_host.numel() * 2 + self.ids_host.numel() * 4 + self.rw_host.numel() * 4)
        self.d2h = T * H * 4
        self.kernels_per_step = 4

    def step(self, i, stream):
        self.w4.w4a16_moe_gemm(self.x, self.ids, self.rw, self.qgu, self.sgu, self.qdn, self.sdn,
                               workspace=self.ws, y=self.y, stream=stream)

    def e2e_step(self, i, stream):
        self.x.copy_(self.x_host, non_blocking=True)
        self.ids.copy_(self.ids_host, non_blocking=True)
        self.rw.copy_(self.rw_host, non_blocking=True)
        self.step(i, stream)
        self.y_host.copy_(self.y, non_blocking=True)
        stream.synchronize()

    def oracle_sample(self, budget_s):
        tokens = [0]
        experts = moe_host_experts(sorted({int(e) for e in self.ids_np[0]}), self.seed, self.dev)
        per_call, desc = oracle_moe_sample(self.x_np, self.ids_np, self.rw_np, experts, tokens)
        return self.bytes / per_call / 1e12, desc


class MoeBlockWorkload(Workload):
    """Whole MoE block on the experts of a MoeWorkload: router (fp32 weights,
    sigmoid gate, top-8 with a selection bias, scale 2.827), the routed
    layer and one shared expert of width 2048; 128 tokens, bf16."""

    def __init__(self, base: MoeWorkload, seed=0, Is=SHARED_I):
        import synth
        w4, torch, dev = base.w4, base.torch, base.dev
        self.w4, self.torch, self.dev, self.base, self.seed = w4, torch, dev, base, seed
        T, H, I, E, topk = base.T, base.H, base.I, base.E, base.topk
        self.T, self.E, self.topk, self.Is = T, E, topk, Is
        self.name = f"MoE block T={T} E={E} top-{topk} + shared expert Is={Is} bf16"
        self.dtype = "bf16"
        self.scale = 2.827
        self.wr = synth.weights_device(seed + 1, E, H, dev)
        bias = synth.activations(seed + 1, 1, E)[0] * np.float32(0.05)
        self.bias_np = bias
        self.bias = torch.from_numpy(bias).to(dev)
        self.shared_w = (synth.weights_device(seed, 2 * Is, H, dev, sub=2 * E),
                         synth.weights_device(seed, H, Is, dev, sub=2 * E + 1))
        self.shared = (w4.w4a16_quantize(self.shared_w[0]) + w4.w4a16_quantize(self.shared_w[1]))
        self.ws = torch.empty(w4.w4a16_moe_block_workspace_size(T, topk, E, H, I, Is),
                              dtype=torch.uint8, device=dev)
        self.y = torch.empty((T, H), dtype=torch.float32, device=dev)
        self.y_host = base.y_host
        # the device routing of this input fixes the active experts
        _, ids, rw = w4.w4a16_moe_route(base.x, self.wr, topk, bias=self.bias,
                                        route_scale=self.scale)
        self.ids_np, self.rw_np = ids.cpu().numpy(), rw.cpu().numpy()
        self.active = len(set(int(e) for e in self.ids_np.reshape(-1)))
        shared_bytes = (2 * Is * H // 2 + 2 * Is * (H // 32) * 4) + (H * Is // 2 + H * (Is // 32) * 4)
        self.bytes = (self.active * base.per_expert + shared_bytes + E * H * 4 + T * H * 2 +
                      T * H * 4)
        self.flops = 2.0 * T * (topk * (2 * I * H + H * I) + (2 * Is * H + H * Is) + E * H)
        self.h2d = base.x_host.numel() * 2
        self.d2h = T * H * 4
        self.kernels_per_step = (2 + w4.w4a16_gemm_launches(T, 2 * Is, H, "bf16") + 1 +
                                 w4.w4a16_gemm_launches(T, H, Is, "bf16") + 4)

    def step(self, i, stream):
        b = self.base
        self.w4.w4a16_moe_block(b.x, self.wr, self.topk, b.qgu, b.sgu, b.qdn, b.sdn,
                                shared=self.shared, bias=self.bias, route_scale=self.scale,
                                workspace=self.ws, y=self.y, stream=stream)

    def e2e_step(self, i, stream):
        self.base.x.copy_(self.base.x_host, non_blocking=True)
        self.step(i, stream)
        self.y_host.copy_(self.y, non_blocking=True)
        stream.synchronize()

    def oracle_sample(self, budget_s):
        import oracle
        tokens = [0]
        experts = moe_host_experts(sorted({int(e) for e in self.ids_np[0]}), self.seed, self.dev)
        shared = (oracle.quantize_w4a16(self.shared_w[0].cpu().numpy()) +
                  oracle.quantize_w4a16(self.shared_w[1].cpu().numpy()))
        router = (self.wr.cpu().numpy(), self.bias_np, self.topk, self.scale)
        per_call, desc = oracle_moe_sample(self.base.x_np, self.ids_np, self.rw_np, experts,
                                           tokens, shared=shared, router=router)
        return self.bytes / per_call / 1e12, desc


def make_workloads(keys, w4, torch, dev, overlap=True, moe_experts=MOE_E, moe_tokens=MOE_T,
                   algo="auto"):
    out = {}
    moe = None
    for key in keys:
        if key in GEMM_SPECS:
            M, N, K, dt, seed, outlier, name = GEMM_SPECS[key]
            out[key] = GemmWorkload(w4, torch, dev, M, N, K, dt, seed, outlier, algo=algo,
                                    overlap=overlap, name=name)
        elif key in ("2-f32", "2-bf16"):
            out[key] = PairWorkload(w4, torch, dev, key.split("-")[1], overlap=overlap)
        elif key in ("3", "5"):
            if moe is None:
                moe = MoeWorkload(w4, torch, dev, T=moe_tokens, E=moe_experts)
            out[key] = moe if key == "3" else MoeBlockWorkload(moe)
        else:
            raise ValueError(key)
        out[key].key = key
    return out


# ----------------------------------------------------------------- distributed
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(torch, value, world):
    """Max of `value` over the ranks (the slowest replica sets the time)."""
    if world == 1:
        return value
    import torch.distributed as dist
    dev = "cpu" if dist.get_backend() == "gloo" else "cuda"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(world, units_per_rank_step, max_seconds_per_step):
    """Whole-job rate: every rank's units of one step over the slowest rank's
    time (replicas: per-rank work is fixed as N grows, "weak" scaling)."""
    return world * units_per_rank_step / max_seconds_per_step


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------- timing
def time_graph(torch, steps_fn, steps, warmup, stream, world=1, step_offset=0):
    """Warm up eagerly, capture `steps` steps in one graph, replay it once
    between barrier + synchronize; -> (ms, sm_mhz from the device clock probes)."""
    with torch.cuda.stream(stream):
        for i in range(warmup):
            steps_fn(i, stream)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(steps):
            steps_fn(step_offset + warmup + i, torch.cuda.current_stream())
    graph.replay()  # settles the graph upload
    stream.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    barrier(world)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        # hold the stream while the host enqueues the rest, then probe the clock
        torch.cuda._sleep(HOLD_CYCLES)
        ev[0].record(stream)
        torch.cuda._sleep(CLOCK_PROBE_CYCLES)
        ev[1].record(stream)
        ev[2].record(stream)
        graph.replay()
        ev[3].record(stream)
        ev[4].record(stream)
        torch.cuda._sleep(CLOCK_PROBE_CYCLES)
        ev[5].record(stream)
    stream.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    ms = ev[2].elapsed_time(ev[3])
    mhz = [CLOCK_PROBE_CYCLES / (ev[0].elapsed_time(ev[1]) * 1e3),
           CLOCK_PROBE_CYCLES / (ev[4].elapsed_time(ev[5]) * 1e3)]
    del graph
    return ms, mhz


def time_eager_launches(torch, wl, n, stream):
    """Median device time of single eager launches of one step (M=1 per
    launch: programmatic launch has nothing to overlap with here)."""
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n)]
    with torch.cuda.stream(stream):
        for i in range(n):
            torch.cuda._sleep(HOLD_CYCLES // 10)
            ev[2 * i].record(stream)
            wl.step(i, stream)
            ev[2 * i + 1].record(stream)
    stream.synchronize()
    return statistics.median(ev[2 * i].elapsed_time(ev[2 * i + 1]) * 1e3 for i in range(n))


def roofline(wl, per_step_s, pk, traffic_key):
    if wl.bound == "tensor":
        peak = pk["bf16_tflops"]
        factor = getattr(wl, "tensor_factor", 1.0)
        achieved = factor * wl.flops / per_step_s / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s"}
        if factor != 1.0:
            roof["flops"] = "3 x 2MNK: bf16 tensor work of the three activation pieces"
    else:
        peak = pk["hbm_gbs"]
        achieved = wl.bytes / per_step_s / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["peak_source"] = pk["source"]
    roof["traffic"] = profiled_traffic(traffic_key)
    roof["kernels_per_step"] = wl.kernels_per_step
    return roof


def measure(torch, wl, args, stream, pk, world=1, e2e_steps=None, cpu_budget=None):
    """Device time, roofline, e2e and CPU baseline of one workload."""
    ms, mhz = time_graph(torch, wl.step, args.steps, args.warmup, stream, world)
    ms = reduce_max(torch, ms, world)
    per_step_s = ms / 1e3 / args.steps
    r = {
        "workload": wl.name,
        "value": aggregate_rate(world, wl.flops if wl.unit == "TFLOP/s" else wl.bytes,
                                per_step_s) / 1e12,
        "unit": wl.unit, "ms_per_step": ms / args.steps, "us_per_call": per_step_s * 1e6,
        "dtype": wl.dtype, "gpu_launches": wl.kernels_per_step * args.steps,
        "sm_mhz_device": [round(v, 1) for v in mhz],
        "roofline": roofline(wl, per_step_s, pk, traffic_key(wl.key)),
    }
    if isinstance(wl, PairWorkload):
        per = {}
        for p in wl.parts:
            pms, _ = time_graph(torch, p.step, args.steps, args.warmup, stream, world,
                                step_offset=1000)
            ps = reduce_max(torch, pms, world) / 1e3 / args.steps
            pr = roofline(p if wl.bound == "hbm" else _Scaled(p, wl.tensor_factor), ps, pk, None)
            pr.pop("traffic")
            per[p.name] = {"shape": f"{p.M}x{p.K}->{p.N}", "us_per_call": ps * 1e6,
                           "roofline": pr}
        r["kernels"] = per
    if getattr(wl, "M", 0) == 1:
        r["eager_us_per_launch"] = time_eager_launches(torch, wl, 50, stream)
    if e2e_steps:
        with torch.cuda.stream(stream):
            wl.e2e_step(0, stream)
            barrier(world)
            t0 = time.perf_counter()
            for i in range(e2e_steps):
                wl.e2e_step(i, stream)
            t_e2e = time.perf_counter() - t0
        per_e2e = reduce_max(torch, t_e2e, world) / e2e_steps
        r["e2e"] = {"value": aggregate_rate(world, wl.flops if wl.unit == "TFLOP/s" else wl.bytes,
                                            per_e2e) / 1e12,
                    "unit": wl.unit, "h2d_bytes_per_step": wl.h2d, "d2h_bytes_per_step": wl.d2h,
                    "steps": e2e_steps}
    if cpu_budget:
        v, desc = wl.oracle_sample(cpu_budget)
        r["cpu_baseline"] = {"value": v, "unit": wl.unit, "cores": len(os.sched_getaffinity(0)),
                             "kind": "oracle", "sample": desc}
    return r


class _Scaled:
    """A GEMM part seen with the tensor-work factor of its pair."""

    def __init__(self, p, factor):
        self.bound, self.flops, self.bytes = "tensor", p.flops, p.bytes
        self.tensor_factor, self.kernels_per_step = factor, p.kernels_per_step


def traffic_key(key):
    return {"2-f32": "config2_f32", "2-bf16": "config2_bf16"}.get(key, f"config{key}")


# ----------------------------------------------------------------- arms
def run_reference(args):
    """The oracle as the reference arm: K steps, each a bounded sample of the
    headline workload. It never imports the CUDA library."""
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    key = str(args.config)
    budget = max(0.02, min(5.0, 90.0 / max(1, args.steps + args.warmup)))
    if key in GEMM_SPECS or key in ("2-f32", "2-bf16"):
        if key in GEMM_SPECS:
            M, N, K, dt, seed, outlier, _ = GEMM_SPECS[key]
            parts = [(M, N, K, dt, seed, outlier)]
        else:
            dt = key.split("-")[1]
            parts = [(M, N, K, dt, seed, 0.01) for M, N, K, seed, _ in PAIR_SPEC]
        inputs = [gemm_host_inputs(*p) for p in parts]
        nbytes = sum(_gemm_bytes(p[0], p[1], p[2], 2 if p[3] == "bf16" else 4) for p in parts)
        flops = sum(2.0 * p[0] * p[1] * p[2] for p in parts)
        unit = "TFLOP/s" if parts[0][0] >= 1024 else "TB/s"

        def sample():
            secs, descs = 0.0, []
            for x, w in inputs:
                s, d = oracle_gemm_sample(x, w, budget / len(inputs))
                secs += s
                descs.append(d)
            return secs, "; ".join(descs)
    else:
        import torch
        if not torch.cuda.is_available():
            print(json.dumps({"impl": "reference", "unavailable":
                              "the MoE workloads draw their weights with the CUDA generator"}))
            return 0
        import synth
        dev = torch.device("cuda", 0)
        x = _bf16_round(synth.activations(0, MOE_T, MOE_H))
        ids, rw = synth.routing(0, MOE_T, MOE_TOPK, MOE_E)
        experts = moe_host_experts(sorted({int(e) for e in ids[0]}), 0, dev)
        active = len(set(int(e) for e in ids.reshape(-1)))
        per_expert = (2 * MOE_I * MOE_H // 2 + 2 * MOE_I * (MOE_H // 32) * 4) + (
            MOE_H * MOE_I // 2 + MOE_H * (MOE_I // 32) * 4)
        nbytes = active * per_expert + MOE_T * MOE_H * 6
        flops = 2.0 * MOE_T * MOE_TOPK * 3 * MOE_I * MOE_H
        unit = "TB/s"
        if key == "5":
            print(json.dumps({"impl": "reference", "unavailable":
                              "the MoE block's routing comes from the device router"}))
            return 0

        def sample():
            return oracle_moe_sample(x, ids, rw, experts, [0])
    vals, desc = [], ""
    for i in range(args.warmup + args.steps):
        secs, desc = sample()
        if i >= args.warmup:
            vals.append(secs)
    per_step_s = float(np.mean(vals))
    value = (flops if unit == "TFLOP/s" else nbytes) / per_step_s / 1e12
    cores = len(os.sched_getaffinity(0))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": unit,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": per_step_s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded, same draws as the GPU arm)",
        "config": {**workload_config(key), "parallelism": f"replicas x{world}"},
        "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    import int4_w4a16_group_gemm_gb300 as w4

    head = str(args.config)
    extra = [] if (args.only or world > 1) else [k for k in args.configs.split(",") if k and k != head]
    pk = peaks()
    stream = torch.cuda.Stream(device=dev)

    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
    wls = make_workloads([head], w4, torch, dev, overlap=not args.no_overlap,
                         moe_experts=args.moe_experts, moe_tokens=args.moe_tokens,
                         algo=args.algo)
    wl = wls[head]
    res = measure(torch, wl, args, stream, pk, world, e2e_steps=min(args.steps, args.e2e_steps),
                  cpu_budget=None)
    clocks = sampler.stop() if sampler else None
    status = w4.w4a16_last_device_status(stream)
    if status != 0:
        raise RuntimeError(f"device status after the timed region: {w4.status_string(status)}")

    line = {
        "metric": METRIC, "value": res["value"], "unit": wl.unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": wl.dtype,
        "data": "synthetic (seeded: x ~ N(0,1), W ~ N(0,1/K) quantised on the device)",
        "config": {**workload_config(head, args.moe_experts, args.moe_tokens),
                   "parallelism": f"replicas x{world}",
                   **({"algo": args.algo} if args.algo != "auto" else {})},
        "timing": {"method": ("one CUDA graph of K steps, replayed once; stream held by a spin "
                              "kernel before the start event (host enqueue time not counted)"),
                   "overlap": not args.no_overlap, "us_per_call": res["us_per_call"],
                   "sm_mhz_device": res["sm_mhz_device"],
                   **({"eager_us_per_launch": res["eager_us_per_launch"]}
                      if "eager_us_per_launch" in res else {})},
        "roofline": res["roofline"],
        "e2e": res["e2e"],
        "gpu_launches": res["gpu_launches"],
        "clocks": clocks,
    }
    if "kernels" in res:
        line["kernels"] = res["kernels"]
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, desc = wl.oracle_sample(args.cpu_budget)
        line["cpu_baseline"] = {"value": v, "unit": wl.unit,
                                "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
                                "sample": desc}
    if extra:
        configs = {}
        others = make_workloads(extra, w4, torch, dev, overlap=not args.no_overlap,
                                moe_experts=args.moe_experts, moe_tokens=args.moe_tokens,
                                algo=args.algo)
        csampler = ClockSampler(local)
        csampler.start()
        for key in extra:
            r = measure(torch, others[key], args, stream, pk, world,
                        e2e_steps=min(args.steps, 20),
                        cpu_budget=None if args.no_cpu_baseline else args.cpu_budget_configs)
            r["config"] = workload_config(key, args.moe_experts, args.moe_tokens)
            configs[key] = r
        cclocks = csampler.stop()
        if w4.w4a16_last_device_status(stream) != 0:
            raise RuntimeError("device status after the configs sweep")
        line["configs"] = configs
        line["configs_clocks"] = cclocks
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="1", choices=ALL_CONFIGS,
                    help="headline workload (default: the decode GEMV)")
    ap.add_argument("--configs", default=",".join(ALL_CONFIGS),
                    help="workloads measured after the headline (comma list)")
    ap.add_argument("--only", action="store_true", help="measure the headline workload only")
    ap.add_argument("--no-overlap", action="store_true",
                    help="launch without programmatic dependent launch (W4A16_FLAG_OVERLAP)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--cpu-budget-configs", type=float, default=3.0)
    ap.add_argument("--e2e-steps", type=int, default=2000)
    ap.add_argument("--moe-experts", type=int, default=MOE_E,
                    help="experts of the MoE workloads (configs 3 and 5); fewer only to profile "
                         "the same kernels on a smaller working set")
    ap.add_argument("--algo", default="auto", choices=["auto", "stream", "gemv", "tc"],
                    help="GEMM kernel of the single-GEMM workloads (configs 0, 1, 4); auto "
                         "is the library's own choice")
    ap.add_argument("--moe-tokens", type=int, default=MOE_T,
                    help="tokens of the MoE workloads (configs 3 and 5); see --moe-experts")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
