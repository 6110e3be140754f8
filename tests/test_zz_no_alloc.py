"""w4a16_moe_gemm_noalloc: the MoE entry point for callers that cannot
allocate device memory (for example serving processes that reserve their
whole budget at start-up, or plugins whose host framework owns every
allocation and offers no workspace). It keeps its intermediates in a fixed
40 MiB array inside the library instead of a caller workspace.

Checked through the C ABI against the workspace entry point on the same
inputs, on two calls in a row (the second call finds the first call's
leftovers in the shared array). Both outputs must be within the MoE
tolerance the other tests use (the oracle's propagated bound) of the
workspace entry point's output and of the oracle's; the kernels are
deterministic, so they are expected to be bit-identical to the former.
Sizes whose intermediates exceed the array are rejected.

This file is collected last so a run that stops at the first failure has
run every other test before it; it also passes alone in a fresh process.
"""

import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w4():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import int4_w4a16_group_gemm_gb300 as w4
    return w4


def device_experts(w4, seed, E, H, I):
    dev = torch.device("cuda")
    qgu = torch.empty((E, 2 * I, H // 8), dtype=torch.int32, device=dev)
    sgu = torch.empty((E, 2 * I, H // 32), dtype=torch.float32, device=dev)
    qdn = torch.empty((E, H, I // 8), dtype=torch.int32, device=dev)
    sdn = torch.empty((E, H, I // 32), dtype=torch.float32, device=dev)
    for e in range(E):
        w4.w4a16_quantize(synth.weights_device(seed, 2 * I, H, dev, sub=2 * e), qw=qgu[e], sc=sgu[e])
        w4.w4a16_quantize(synth.weights_device(seed, H, I, dev, sub=2 * e + 1), qw=qdn[e], sc=sdn[e])
    return qgu, sgu, qdn, sdn


@pytest.mark.parametrize("T,H,I,E,topk,bf16", [
    (16, 1024, 512, 9, 4, True),
    (5, 256, 128, 6, 2, False),
    (128, 7168, 2048, 16, 8, True),   # near the array's limit (~37.4 MB of intermediates)
])
def test_noalloc_matches_workspace_entry_point(w4, T, H, I, E, topk, bf16):
    seed = 11 + T + E
    x = synth.activations(seed, T, H)
    ids, rw = synth.routing(seed, T, topk, E)
    xt = torch.from_numpy(x)
    if bf16:
        xt = xt.to(torch.bfloat16)
    xd, idd, rwd = xt.cuda(), torch.from_numpy(ids).cuda(), torch.from_numpy(rw).cuda()
    experts = device_experts(w4, seed, E, H, I)
    assert w4.w4a16_moe_workspace_size(T, topk, E, H, I) <= 40 << 20

    y_ws = w4.w4a16_moe_gemm(xd, idd, rwd, *experts)
    y1 = w4.w4a16_moe_gemm_noalloc(xd, idd, rwd, *experts)
    y2 = w4.w4a16_moe_gemm_noalloc(xd, idd, rwd, *experts)
    torch.cuda.synchronize()
    assert w4.w4a16_last_device_status() == w4.W4A16_OK

    # tolerance of the MoE tests: the oracle's propagated bound, on the
    # tokens it can afford to recompute; the oracle quantises the experts
    # itself from the same seeded draws
    tokens = list(range(min(T, 3)))
    used = sorted({int(e) for t in tokens for e in ids[t]})
    dev = torch.device("cuda")
    host = {}
    for e in used:
        wg = synth.weights_device(seed, 2 * I, H, dev, sub=2 * e).cpu().numpy()
        wd = synth.weights_device(seed, H, I, dev, sub=2 * e + 1).cpu().numpy()
        host[e] = oracle.quantize_w4a16(wg) + oracle.quantize_w4a16(wd)
    ref_o, tol = oracle.moe_ref(xt.float().numpy(), ids, rw, {e: v[0] for e, v in host.items()},
                                {e: v[1] for e, v in host.items()},
                                {e: v[2] for e, v in host.items()},
                                {e: v[3] for e, v in host.items()}, bf16,
                                eps=4e-3 if bf16 else 1e-5, tokens=tokens)
    ref = y_ws.cpu().numpy().astype(np.float64)
    for y in (y1, y2):
        got = y.cpu().numpy().astype(np.float64)
        for t in tokens:
            assert np.all(np.abs(got[t] - ref[t]) <= tol[t])
            assert np.all(np.abs(got[t] - ref_o[t]) <= tol[t])
        assert torch.equal(y.view(torch.int32), y_ws.view(torch.int32))


def test_noalloc_rejects_sizes_beyond_the_array(w4):
    lib = w4.lib
    import ctypes
    fake = ctypes.c_void_p(0x1000)
    null = ctypes.c_void_p(0)
    # 4096 tokens x top-8 at hidden 7168 need far more than 40 MiB
    assert w4.w4a16_moe_workspace_size(4096, 8, 384, 7168, 2048) > 40 << 20
    code = lib.w4a16_moe_gemm_noalloc(fake, 1, fake, fake, 4096, 8, fake, fake, fake, fake,
                                      384, 7168, 2048, 32, fake, null)
    assert code == w4.W4A16_ERR_UNSUPPORTED
