"""The bounds-checking build (W4A16_DEBUG, libw4a16_debug.so): every kernel
checks the indices it computes against its buffers and, instead of making an
out-of-bounds access, records W4A16_ERR_BOUNDS in the status word and skips
it. The test builds that library, runs ragged and edge shapes of every entry
point through it and through the release build (each in a child process, one
library per process), and requires a clean status after every call and
output bits identical to the release build's: the checks change no
arithmetic."""

import os
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (M, N, K, activations, algo, group, bf16 output)
GEMM_CASES = [
    (1, 4096, 7168, "f32", "gemv", 32, False),
    (1, 153, 8192, "bf16", "gemv", 32, False),
    (1, 300, 96, "f32", "stream", 32, False),
    (3, 513, 4224, "f32", "stream", 64, False),
    (2, 1000, 2048, "bf16", "stream", 128, True),
    (64, 4096, 7168, "bf16", "tc", 32, False),
    (31, 40, 4224, "bf16", "tc", 64, False),
    (300, 300, 7168, "bf16", "tc", 128, True),
    (257, 513, 160, "bf16", "tc", 32, False),
    (600, 2100, 160, "bf16", "tc", 32, False),
    (17, 1000, 4224, "f32", "tc", 32, False),
    (64, 700, 1024, "f32", "tc", 64, True),
]
# (T, topk, E, H, I, activations)
MOE_CASES = [
    (16, 2, 8, 256, 128, "f32"),
    (37, 4, 11, 512, 256, "bf16"),
    (5, 8, 64, 384, 192, "bf16"),
]


def run_cases(out_path: str) -> None:
    """Child process: run every case through the library that W4A16_LIBRARY
    selects; save outputs and the status after each call."""
    sys.path.insert(0, ROOT)
    import torch

    import int4_w4a16_group_gemm_gb300 as w4
    import synth

    out, status = {}, {}

    def record(name, tensor):
        status[name] = w4.w4a16_last_device_status()
        t = tensor.detach()
        out[name] = (t.view(torch.int16) if t.dtype == torch.bfloat16 else t).cpu().numpy()

    for i, (M, N, K, dt, algo, group, obf) in enumerate(GEMM_CASES):
        x = torch.from_numpy(synth.activations(40 + i, M, K)).cuda()
        if dt == "bf16":
            x = x.to(torch.bfloat16)
        qw, sc = w4.w4a16_quantize(torch.from_numpy(synth.weights(40 + i, N, K)).cuda(),
                                   group=group)
        record(f"quantize{i}", qw)
        y = w4.w4a16_gemm(x, qw, sc, group=group, algo=algo, out_dtype="bf16" if obf else "f32")
        record(f"gemm{i}", y)

    for i, (T, topk, E, H, I, dt) in enumerate(MOE_CASES):
        x = torch.from_numpy(synth.activations(60 + i, T, H)).cuda()
        if dt == "bf16":
            x = x.to(torch.bfloat16)
        ids, rw = synth.routing(60 + i, T, topk, E)
        ids = torch.from_numpy(ids).cuda()
        rw = torch.from_numpy(rw).cuda()
        qgu, sgu = w4.w4a16_quantize(
            torch.from_numpy(synth.weights(60 + i, E * 2 * I, H)).cuda())
        qdn, sdn = w4.w4a16_quantize(torch.from_numpy(synth.weights(61 + i, E * H, I)).cuda())
        qgu, sgu = qgu.view(E, 2 * I, H // 8), sgu.view(E, 2 * I, H // 32)
        qdn, sdn = qdn.view(E, H, I // 8), sdn.view(E, H, I // 32)
        record(f"moe{i}", w4.w4a16_moe_gemm(x, ids, rw, qgu, sgu, qdn, sdn))
        record(f"moe_noalloc{i}", w4.w4a16_moe_gemm_noalloc(x, ids, rw, qgu, sgu, qdn, sdn))
        router_w = torch.from_numpy(synth.weights(62 + i, E, H)).cuda()
        y, bids, brw = w4.w4a16_moe_block(x, router_w, topk, qgu, sgu, qdn, sdn)
        record(f"moe_block{i}", y)
        record(f"moe_block_ids{i}", bids)
        record(f"moe_block_rw{i}", brw)
    np.savez(out_path, **out, **{f"status_{k}": np.array(v) for k, v in status.items()})


torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def debug_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sys.path.insert(0, ROOT)
    from int4_w4a16_group_gemm_gb300 import build
    srcs = build.sources() + [os.path.join(build.CSRC, f) for f in os.listdir(build.CSRC)]
    newest = max(os.path.getmtime(s) for s in srcs)
    if not os.path.exists(build.LIB_DEBUG) or os.path.getmtime(build.LIB_DEBUG) < newest:
        build.build(debug=True)
    return build.LIB_DEBUG


def _run_child(tmp_path, name, lib):
    out = str(tmp_path / f"{name}.npz")
    env = dict(os.environ)
    if lib is None:
        env.pop("W4A16_LIBRARY", None)
    else:
        env["W4A16_LIBRARY"] = lib
    r = subprocess.run([sys.executable, os.path.abspath(__file__), out], env=env, cwd=ROOT,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    return dict(np.load(out))


def test_bounds_checked_build_is_clean_and_bit_identical(debug_lib, tmp_path):
    release = _run_child(tmp_path, "release", None)
    debug = _run_child(tmp_path, "debug", debug_lib)
    assert set(release) == set(debug)
    for k in sorted(debug):
        if k.startswith("status_"):
            assert int(debug[k]) == 0, f"{k[7:]}: status {int(debug[k])} in the checked build"
            assert int(release[k]) == 0, f"{k[7:]}: status {int(release[k])}"
        else:
            assert debug[k].dtype == release[k].dtype and debug[k].shape == release[k].shape, k
            assert np.array_equal(debug[k].view(np.uint8), release[k].view(np.uint8)), k


if __name__ == "__main__":
    run_cases(sys.argv[1])
