"""Benchmark of the W4A16 group-quantised GEMM library on one GB300.

Default workload (the headline): the decode GEMV, M=1, K=7168, N=4096
(fused gate+up of an MoE expert), group 32, fp32 activations, weights
W ~ N(0, 1/K) quantised on the device. A step is one w4a16_gemm call; the
metric is effective TB/s = algorithmic bytes (packed weights + scales +
activations + output) / time.

Other workloads are selectable with --config for the design notes:
  0 tiny GEMM 1x256 -> 512 fp32             (TB/s)
  1 decode GEMV 1x7168 -> 4096 fp32          (TB/s, default)
  2 tree-verify pair M=64 (7168->4096 then 2048->7168), --dtype f32|bf16
  3 grouped MoE layer: 128 tokens, 384 experts, top-8, bf16  (TB/s of
    active-expert bytes)
  4 prefill GEMM 2048x7168 -> 18432 bf16     (TFLOP/s)
  5 whole MoE block: config 3 plus the router and one shared expert
    (width 2048), bf16                       (TB/s of active bytes)

Timing: W warm-up steps, then exactly K steps captured in one CUDA graph
and replayed once between barrier + synchronize, timed with CUDA events on
the launching stream; max over ranks. Working sets below the L2 size rotate
through enough weight copies that every step reads its weights from HBM.
`e2e` repeats the K steps through the Python binding with the per-step
activations copied in from pinned host memory and the result copied back
and waited for. The oracle (CPU, numpy fp64) is timed on a bounded sample
of the same workload as the reported CPU baseline; `--impl reference` runs
that oracle as the reference arm.

Multi-GPU: independent replicas (the path is not partitioned across GPUs);
value = all ranks' bytes / max time, scaling "weak".
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
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
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, ln in self.lines:
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


# ----------------------------------------------------------------- workloads
class Workload:
    """One configuration: device buffers, a step, its bytes and flops."""

    name = ""
    unit = "TB/s"
    dtype = "f32"
    bound = "hbm"

    def step(self, i, stream):
        raise NotImplementedError

    def e2e_step(self, i, stream):
        raise NotImplementedError


def _rotation(bytes_per_copy, l2_bytes):
    return max(1, int(np.ceil(4.0 * l2_bytes / bytes_per_copy)))


class GemmWorkload(Workload):
    def __init__(self, w4, torch, dev, M, N, K, dtype, seed, name, outlier=0.0, algo="auto",
                 l2_bytes=129 * 2 ** 20, overlap=True):
        import synth
        self.w4, self.torch, self.dev = w4, torch, dev
        self.M, self.N, self.K = M, N, K
        self.dtype = dtype
        self.name = name
        self.algo = algo
        self.overlap = overlap
        wbytes = N * K // 2 + N * (K // 32) * 4
        xb = M * K * (2 if dtype == "bf16" else 4)
        self.bytes = wbytes + xb + M * N * 4
        self.flops = 2.0 * M * N * K
        self.ncopies = _rotation(wbytes, l2_bytes) if wbytes < 2 * l2_bytes else 1
        self.qw, self.sc = [], []
        w = synth.weights_device(seed, N, K, dev)
        for c in range(self.ncopies):
            qw, sc = w4.w4a16_quantize(w)
            self.qw.append(qw)
            self.sc.append(sc)
        del w
        x = synth.activations(seed, M, K, outlier_frac=outlier)
        xt = torch.from_numpy(x)
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
        self.kernels_per_step = self._kernels_per_step()

    def _kernels_per_step(self):
        n = self.w4.w4a16_gemm_launches(self.M, self.N, self.K, self.dtype, self.algo)
        if n <= 0:
            raise RuntimeError(f"gemm rejected: status {-n}")
        return n

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
        """Time the oracle on the full problem or a row sample; -> (value, desc)."""
        import oracle
        qw = self.qw[0].cpu().numpy()
        sc = self.sc[0].cpu().numpy()
        x = self.x_host.float().numpy()
        rows = self.N
        t0 = time.perf_counter()
        oracle.gemm_ref(x, qw[:64], sc[:64])
        per_row = (time.perf_counter() - t0) / 64
        rows = int(max(8, min(self.N, budget_s / max(per_row, 1e-9))))
        reps, el = 0, 0.0
        t0 = time.perf_counter()
        while True:
            oracle.gemm_ref(x, qw[:rows], sc[:rows])
            reps += 1
            el = time.perf_counter() - t0
            if el >= budget_s or reps >= 50:
                break
        frac = rows / self.N
        per_call = el / reps / frac
        return self._metric_value(per_call), f"{reps} x oracle.gemm_ref on {rows} of {self.N} weight rows (M={self.M}), scaled to the full call"

    def _metric_value(self, seconds):
        if self.unit == "TFLOP/s":
            return self.flops / seconds / 1e12
        return self.bytes / seconds / 1e12


class TreeVerifyWorkload(Workload):
    """The two M=64 GEMMs of a tree-verify step (7168->4096, 2048->7168)."""

    def __init__(self, w4, torch, dev, dtype, seed=0):
        self.a = GemmWorkload(w4, torch, dev, 64, 4096, 7168, dtype, seed, "a", outlier=0.01)
        self.b = GemmWorkload(w4, torch, dev, 64, 7168, 2048, dtype, seed + 1, "b", outlier=0.01)
        self.name = f"tree-verify pair M=64 (7168->4096, 2048->7168) {dtype}"
        self.dtype = dtype
        self.bytes = self.a.bytes + self.b.bytes
        self.flops = self.a.flops + self.b.flops
        self.h2d = self.a.h2d + self.b.h2d
        self.d2h = self.a.d2h + self.b.d2h
        self.kernels_per_step = self.a.kernels_per_step + self.b.kernels_per_step
        # bf16: HBM-bound on the tensor cores. fp32: the fp32-exact tensor-core
        # kernel multiplies three bf16 pieces of every activation, so its
        # tensor work is 3 x 2MNK, which outweighs the HBM time at M = 64.
        self.bound = "hbm" if dtype == "bf16" else "tensor"
        self.tensor_flops = self.flops if dtype == "bf16" else 3.0 * self.flops

    def step(self, i, stream):
        self.a.step(i, stream)
        self.b.step(i, stream)

    def e2e_step(self, i, stream):
        self.a.e2e_step(i, stream)
        self.b.e2e_step(i, stream)

    def oracle_sample(self, budget_s):
        va, da = self.a.oracle_sample(budget_s / 2)
        vb, db = self.b.oracle_sample(budget_s / 2)
        ta, tb = self.a.bytes / (va * 1e12), self.b.bytes / (vb * 1e12)
        return self.bytes / (ta + tb) / 1e12, f"{da}; {db}"


class MoeWorkload(Workload):
    """Grouped MoE layer: 128 tokens, hidden 7168, 384 experts (I=2048), top-8, bf16."""

    def __init__(self, w4, torch, dev, seed=0, T=128, H=7168, I=2048, E=384, topk=8):
        import synth
        self.w4, self.torch, self.dev = w4, torch, dev
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
        x = synth.activations(seed, T, H)
        ids, rw = synth.routing(seed, T, topk, E)
        self.ids_np, self.rw_np = ids, rw
        self.x_host = torch.from_numpy(x).to(torch.bfloat16).pin_memory()
        self.ids_host = torch.from_numpy(ids).pin_memory()
        self.rw_host = torch.from_numpy(rw).pin_memory()
        self.x = self.x_host.to(dev)
        self.ids = self.ids_host.to(dev)
        self.rw = self.rw_host.to(dev)
        self.ws = torch.empty(w4.w4a16_moe_workspace_size(T, topk, E, H, I), dtype=torch.uint8,
                              device=dev)
        self.y = torch.empty((T, H), dtype=torch.float32, device=dev)
        self.y_host = torch.empty((T, H), dtype=torch.float32).pin_memory()
        active = len(set(int(e) for e in ids.reshape(-1)))
        self.active = active
        per_expert = (2 * I * H // 2 + 2 * I * (H // 32) * 4) + (H * I // 2 + H * (I // 32) * 4)
        self.bytes = active * per_expert + T * H * 2 + T * H * 4
        self.flops = 2.0 * T * topk * (2 * I * H + H * I)
        self.h2d = (self.x_host.numel() * 2 + self.ids_host.numel() * 4 + self.rw_host.numel() * 4)
        self.d2h = T * H * 4
        self.kernels_per_step = 4
        self.bound = "hbm"
        self.unit = "TB/s"

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
        import oracle
        t0 = time.perf_counter()
        tokens = []
        experts = {}
        for t in range(self.T):
            tokens.append(t)
            for e in self.ids_np[t]:
                e = int(e)
                if e not in experts:
                    experts[e] = (self.qgu[e].cpu().numpy(), self.sgu[e].cpu().numpy(),
                                  self.qdn[e].cpu().numpy(), self.sdn[e].cpu().numpy())
            if len(tokens) >= 2:
                break
        x = self.x_host.float().numpy()
        t1 = time.perf_counter()
        oracle.moe_ref(x, self.ids_np, self.rw_np, {e: v[0] for e, v in experts.items()},
                       {e: v[1] for e, v in experts.items()}, {e: v[2] for e, v in experts.items()},
                       {e: v[3] for e, v in experts.items()}, True, eps=4e-3, tokens=tokens)
        el = time.perf_counter() - t1
        # scale: the full layer touches every active expert once per token-slot
        per_pair = el / (len(tokens) * self.topk)
        full = per_pair * self.T * self.topk
        return self.bytes / full / 1e12, (f"oracle.moe_ref on {len(tokens)} tokens "
                                          f"({len(experts)} experts), scaled by token-slots")


class MoeBlockWorkload(MoeWorkload):
    """Whole MoE block: router (fp32 weights, sigmoid gate, top-8 of 384 with
    a selection bias, scale 2.827), the routed layer of MoeWorkload and one
    shared expert of width 2048; 128 tokens, hidden 7168, bf16."""

    def __init__(self, w4, torch, dev, seed=0, T=128, H=7168, I=2048, E=384, topk=8, Is=2048):
        import synth
        super().__init__(w4, torch, dev, seed, T, H, I, E, topk)
        self.name = (f"MoE block T={T} H={H} I={I} E={E} top-{topk} + shared expert "
                     f"Is={Is}, router fp32, bf16")
        self.Is = Is
        self.scale = 2.827
        self.wr = synth.weights_device(seed + 1, E, H, dev)
        bias = synth.activations(seed + 1, 1, E)[0] * np.float32(0.05)
        self.bias_np = bias
        self.bias = torch.from_numpy(bias).to(dev)
        self.shared = (w4.w4a16_quantize(synth.weights_device(seed, 2 * Is, H, dev, sub=2 * E)) +
                       w4.w4a16_quantize(synth.weights_device(seed, H, Is, dev, sub=2 * E + 1)))
        self.ws = torch.empty(w4.w4a16_moe_block_workspace_size(T, topk, E, H, I, Is),
                              dtype=torch.uint8, device=dev)
        # the device routing of this input fixes the active experts
        _, ids, rw = w4.w4a16_moe_route(self.x, self.wr, topk, bias=self.bias,
                                        route_scale=self.scale)
        self.ids_np, self.rw_np = ids.cpu().numpy(), rw.cpu().numpy()
        active = len(set(int(e) for e in self.ids_np.reshape(-1)))
        self.active = active
        per_expert = (2 * I * H // 2 + 2 * I * (H // 32) * 4) + (H * I // 2 + H * (I // 32) * 4)
        shared_bytes = (2 * Is * H // 2 + 2 * Is * (H // 32) * 4) + (H * Is // 2 + H * (Is // 32) * 4)
        self.bytes = (active * per_expert + shared_bytes + E * H * 4 + T * H * 2 + T * H * 4)
        self.flops = 2.0 * T * (topk * (2 * I * H + H * I) + (2 * Is * H + H * Is) + E * H)
        self.h2d = self.x_host.numel() * 2
        self.d2h = T * H * 4
        self.kernels_per_step = (2 + w4.w4a16_gemm_launches(T, 2 * Is, H, "bf16") + 1 +
                                 w4.w4a16_gemm_launches(T, H, Is, "bf16") + 4)

    def step(self, i, stream):
        self.w4.w4a16_moe_block(self.x, self.wr, self.topk, self.qgu, self.sgu, self.qdn, self.sdn,
                                shared=self.shared, bias=self.bias, route_scale=self.scale,
                                workspace=self.ws, y=self.y, stream=stream)

    def e2e_step(self, i, stream):
        self.x.copy_(self.x_host, non_blocking=True)
        self.step(i, stream)
        self.y_host.copy_(self.y, non_blocking=True)
        stream.synchronize()

    def oracle_sample(self, budget_s):
        import oracle
        tokens = [0, 1]
        experts = {}
        for t in tokens:
            for e in self.ids_np[t]:
                e = int(e)
                if e not in experts:
                    experts[e] = (self.qgu[e].cpu().numpy(), self.sgu[e].cpu().numpy(),
                                  self.qdn[e].cpu().numpy(), self.sdn[e].cpu().numpy())
        shared = tuple(v.cpu().numpy() for v in self.shared)
        x = self.x_host.float().numpy()
        wr = self.wr.cpu().numpy()
        t1 = time.perf_counter()
        oracle.moe_route_ref(x[tokens], wr, self.bias_np, self.topk, self.scale)
        oracle.moe_block_ref(x, self.ids_np, self.rw_np, {e: v[0] for e, v in experts.items()},
                             {e: v[1] for e, v in experts.items()},
                             {e: v[2] for e, v in experts.items()},
                             {e: v[3] for e, v in experts.items()}, shared, True, eps=4e-3,
                             tokens=tokens)
        el = time.perf_counter() - t1
        full = el / len(tokens) * self.T
        return self.bytes / full / 1e12, (f"oracle router + moe_block_ref on {len(tokens)} tokens "
                                          f"({len(experts)} experts + shared), scaled by tokens")


def make_workload(cfg, dtype, w4, torch, dev, overlap=True, moe_experts=384, moe_tokens=128):
    if cfg == 0:
        return GemmWorkload(w4, torch, dev, 1, 512, 256, "f32", 0, "tiny GEMM M=1 K=256 N=512 fp32",
                            overlap=overlap)
    if cfg == 1:
        return GemmWorkload(w4, torch, dev, 1, 4096, 7168, "f32", 0,
                            "decode GEMV M=1 K=7168 N=4096 group=32 fp32 activations",
                            overlap=overlap)
    if cfg == 2:
        return TreeVerifyWorkload(w4, torch, dev, dtype)
    if cfg == 3:
        return MoeWorkload(w4, torch, dev, T=moe_tokens, E=moe_experts)
    if cfg == 4:
        return GemmWorkload(w4, torch, dev, 2048, 18432, 7168, "bf16", 0,
                            "prefill GEMM M=2048 K=7168 N=18432 bf16")
    if cfg == 5:
        return MoeBlockWorkload(w4, torch, dev, T=moe_tokens, E=moe_experts)
    raise ValueError(cfg)


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


# ----------------------------------------------------------------- arms
def run_reference(args):
    """The oracle as the reference arm: K steps, each a bounded sample."""
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import torch
    import int4_w4a16_group_gemm_gb300 as w4
    dev = torch.device("cuda", 0)
    wl = make_workload(args.config, args.dtype, w4, torch, dev, moe_experts=args.moe_experts,
                       moe_tokens=args.moe_tokens)
    budget = max(0.02, min(5.0, 90.0 / max(1, args.steps + args.warmup)))
    vals = []
    desc = ""
    for i in range(args.warmup + args.steps):
        v, desc = wl.oracle_sample(budget)
        if i >= args.warmup:
            vals.append(v)
    value = float(np.mean(vals)) if vals else 0.0
    cores = len(os.sched_getaffinity(0))
    per_step_s = (wl.bytes / (value * 1e12)) if value > 0 and wl.unit == "TB/s" else (
        wl.flops / (value * 1e12) if value > 0 else 0.0)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": wl.unit,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": per_step_s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name},
        "cpu_baseline": {"value": value, "unit": wl.unit, "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": wl.unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
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

    wl = make_workload(args.config, args.dtype, w4, torch, dev, overlap=not args.no_overlap,
                       moe_experts=args.moe_experts, moe_tokens=args.moe_tokens)
    stream = torch.cuda.Stream(device=dev)
    pk = peaks()

    # warm-up (eager)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            wl.step(i, stream)
    stream.synchronize()

    # capture exactly K steps in one graph
    graph = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for i in range(args.steps):
                wl.step(args.warmup + i, torch.cuda.current_stream())
        # one untimed replay to settle the graph upload
        graph.replay()
        stream.synchronize()

    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        if graph is not None:
            graph.replay()
        else:
            for i in range(args.steps):
                wl.step(args.warmup + i, stream)
        ev1.record(stream)
    stream.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    ms = ev0.elapsed_time(ev1)
    clocks = sampler.stop() if sampler else None
    ms = reduce_max(torch, ms, world)
    status = w4.w4a16_last_device_status(stream)
    if status != 0:
        raise RuntimeError(f"device status after the timed region: {w4.status_string(status)}")

    per_step_s = ms / 1e3 / args.steps
    value = aggregate_rate(world, wl.flops if wl.unit == "TFLOP/s" else wl.bytes, per_step_s) / 1e12

    # end to end through the public API, host buffers in and out each step
    e2e_steps = min(args.steps, args.e2e_steps)
    with torch.cuda.stream(stream):
        wl.e2e_step(0, stream)
        barrier(world)
        t0 = time.perf_counter()
        for i in range(e2e_steps):
            wl.e2e_step(i, stream)
        t_e2e = time.perf_counter() - t0
    t_e2e = reduce_max(torch, t_e2e, world)
    per_e2e = t_e2e / e2e_steps
    e2e_value = aggregate_rate(world, wl.flops if wl.unit == "TFLOP/s" else wl.bytes, per_e2e) / 1e12

    # roofline of the dominant kernel (the only kernel of the decode step)
    per_launch_s = per_step_s / wl.kernels_per_step
    if wl.bound == "tensor":
        peak = pk["bf16_tflops"]
        tflops = getattr(wl, "tensor_flops", wl.flops)
        achieved = tflops / wl.kernels_per_step / per_launch_s / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s"}
        if tflops != wl.flops:
            roof["flops"] = "3 x 2MNK: bf16 tensor work of the three activation pieces"
    elif wl.bound == "alu":
        # fp32 FMA peak: 152 SMs x 128 lanes x 2 flop x max SM clock
        peak = 152 * 128 * 2 * 2070e6 / 1e12
        achieved = wl.flops / per_step_s / 1e12
        roof = {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s"}
    else:
        peak = pk["hbm_gbs"]
        achieved = wl.bytes / wl.kernels_per_step / per_launch_s / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["peak_source"] = pk["source"]
    roof["traffic"] = profiled_traffic(
        f"config{args.config}" + (f"_{args.dtype}" if args.config == 2 else ""))

    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": value, "unit": wl.unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": wl.dtype, "data": "synthetic (seeded: x ~ N(0,1), W ~ N(0,1/K) quantised on device)",
        "config": {"workload": wl.name, "config_index": args.config,
                   "l2": (f"{getattr(wl, 'ncopies', 1)} rotating weight copies (> 4x L2)"
                          if getattr(wl, "ncopies", 1) > 1 else "working set larger than L2"),
                   "timing": "one CUDA graph of K steps" if graph is not None else "eager launches",
                   "overlap": bool(getattr(wl, "overlap", False)),
                   "parallelism": f"replicas x{world}",
                   **({"active_experts": wl.active} if hasattr(wl, "active") else {})},
        "roofline": roof,
        "e2e": {"value": e2e_value, "unit": wl.unit, "h2d_bytes_per_step": wl.h2d,
                "d2h_bytes_per_step": wl.d2h, "steps": e2e_steps},
        "gpu_launches": wl.kernels_per_step * args.steps,
        "clocks": clocks,
    }
    if world == 1 and not args.no_cpu_baseline:
        v, desc = wl.oracle_sample(args.cpu_budget)
        line["cpu_baseline"] = {"value": v, "unit": wl.unit,
                                "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
                                "sample": desc}
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=1)
    ap.add_argument("--dtype", choices=["f32", "bf16"], default="bf16")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--no-overlap", action="store_true",
                    help="launch without programmatic dependent launch (W4A16_FLAG_OVERLAP)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--e2e-steps", type=int, default=2000)
    ap.add_argument("--moe-experts", type=int, default=384,
                    help="experts of the MoE workloads (configs 3 and 5); fewer only to profile "
                         "the same kernels on a smaller working set")
    ap.add_argument("--moe-tokens", type=int, default=128,
                    help="tokens of the MoE workloads (configs 3 and 5); see --moe-experts")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
