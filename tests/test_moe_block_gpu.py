"""Parity of the CUDA MoE block (router + routed experts + shared expert)
with the CPU oracle, through the C ABI.

Router: the logits are compared element by element (fp32 accumulation:
within 1e-5 * sum|x * W_r|). The top-k choice is an integer decision taken
from fp32 scores on the device and fp64 scores in the oracle, so the device's
choice is checked for validity against the oracle's scores (every chosen
expert scores at least as high as every unchosen one, up to the score error
the logit tolerance allows) and must equal the oracle's choice wherever the
oracle's k-th and (k+1)-th scores are further apart than that. The weights
are compared for the device's choice.

Block: the device's routing (ids and weights) is fed to the oracle's block,
which adds the shared expert as a last slot of weight 1; every output must be
within the propagated bound of moe_block_ref.

Inputs: x ~ N(0, 1) (fp32, or rounded to bf16), router weights ~ N(0, 1/H)
so that logits are O(1), selection bias ~ 0.05 N(0, 1), experts as in the
grouped-layer tests; the full-size case is the 128-token, hidden 7168, 384
experts of width 2048, top-8 layer with one shared expert of width 2048.
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


def check_route(logits_d, ids_d, w_d, x, wr, bias, topk, scale):
    """Compare a device routing with the oracle's (see the module docstring)."""
    lref, bound, ids_r, _ = oracle.moe_route_ref(x, wr, bias, topk, scale)
    T, E = lref.shape
    ltol = 1e-5 * bound
    err = np.abs(logits_d.astype(np.float64) - lref)
    assert np.all(err <= ltol), f"logits: max err/tol {np.max(err / np.maximum(ltol, 1e-300)):.3e}"
    s = oracle.sigmoid(lref)
    b = np.zeros(E) if bias is None else bias.astype(np.float64)
    sel = s + b
    # score error: sigmoid' <= 1/4 on the logit error, plus the fp32 sigmoid
    ds = 0.25 * ltol + 2.0 ** -21
    for t in range(T):
        chosen = ids_d[t]
        assert len(set(chosen.tolist())) == topk and chosen.min() >= 0 and chosen.max() < E
        mask = np.zeros(E, bool)
        mask[chosen] = True
        slack = 2 * np.max(ds[t])
        if topk < E:
            assert sel[t, mask].min() >= sel[t, ~mask].max() - slack, f"token {t}: invalid top-k"
        # slots in decreasing score order
        assert np.all(np.diff(sel[t, chosen]) <= slack)
        # unique where the oracle's boundary has a margin
        order = np.sort(sel[t])[::-1]
        if topk == E or order[topk - 1] - order[topk] > slack:
            assert set(chosen.tolist()) == set(ids_r[t].tolist()), f"token {t}: not the top-k"
        # weights of the device's choice
        sc = s[t, chosen]
        tot = sc.sum()
        wref = scale * sc / tot
        dsc = ds[t, chosen]
        wtol = abs(scale) * (dsc / tot + sc * dsc.sum() / tot ** 2) * 1.01 + abs(scale) * 2.0 ** -21
        assert np.all(np.abs(w_d[t].astype(np.float64) - wref) <= wtol), f"token {t}: weights"
    return ids_r


def to_dev(a, dt=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dt is not None:
        t = t.to(dt)
    return t.cuda()


@pytest.mark.parametrize("T,E,H,topk,use_bias,dt", [
    (128, 384, 7168, 8, True, "bf16"), (128, 384, 7168, 8, False, "f32"),
    (37, 64, 256, 6, False, "f32"), (5, 1000, 96, 32, True, "f32"), (1, 8, 32, 8, False, "bf16"),
    (300, 160, 512, 1, True, "bf16"),
])
def test_router(w4, T, E, H, topk, use_bias, dt):
    seed = T + E + H
    x = synth.activations(seed, T, H)
    xt = torch.from_numpy(x)
    if dt == "bf16":
        xt = xt.to(torch.bfloat16)
    wr = synth.weights(seed, E, H, sub=1)
    bias = (synth.activations(seed, 1, E, outlier_frac=0.0)[0] * np.float32(0.05)) if use_bias else None
    logits, ids, rw = w4.w4a16_moe_route(xt.cuda(), to_dev(wr), topk,
                                         bias=to_dev(bias) if use_bias else None, route_scale=2.5)
    torch.cuda.synchronize()
    assert w4.w4a16_last_device_status() == w4.W4A16_OK
    check_route(logits.cpu().numpy(), ids.cpu().numpy(), rw.cpu().numpy(), xt.float().numpy(), wr,
                bias, topk, 2.5)


def test_router_ties_go_to_the_lower_id(w4):
    T, E, H, topk = 4, 16, 64, 3
    x = np.abs(synth.activations(3, T, H))
    wr = np.zeros((E, H), np.float32)
    wr[:] = synth.weights(3, E, H) * np.float32(0.1)
    wr[9] = wr[3] = np.float32(1.0)            # the two largest logits, bit-identical
    _, ids, rw = w4.w4a16_moe_route(to_dev(x), to_dev(wr), topk)
    ids = ids.cpu().numpy()
    rw = rw.cpu().numpy()
    assert np.all(ids[:, 0] == 3) and np.all(ids[:, 1] == 9)
    assert np.all(rw[:, 0] == rw[:, 1])


def build_experts(seed, E, H, I, group):
    qgu, sgu, qdn, sdn = [], [], [], []
    for e in range(E):
        a, b = oracle.quantize_w4a16(synth.weights(seed, 2 * I, H, sub=2 * e), group)
        c, d = oracle.quantize_w4a16(synth.weights(seed, H, I, sub=2 * e + 1), group)
        qgu.append(a); sgu.append(b); qdn.append(c); sdn.append(d)
    return np.stack(qgu), np.stack(sgu), np.stack(qdn), np.stack(sdn)


@pytest.mark.parametrize("T,H,I,Is,E,topk,dt,group", [
    (5, 256, 128, 128, 6, 2, "f32", 32), (5, 256, 128, 128, 6, 2, "bf16", 32),
    (16, 1024, 256, 512, 9, 4, "bf16", 64), (40, 512, 128, 256, 4, 1, "f32", 32),
    (70, 256, 128, 128, 8, 3, "f32", 128), (3, 256, 128, 0, 5, 2, "bf16", 32),
    (64, 512, 256, 256, 12, 8, "bf16", 32),
])
def test_small_block(w4, T, H, I, Is, E, topk, dt, group):
    seed = T + H + E + Is
    x = synth.activations(seed, T, H)
    xt = torch.from_numpy(x)
    if dt == "bf16":
        xt = xt.to(torch.bfloat16)
    wr = synth.weights(seed, E, H, sub=100)
    bias = synth.activations(seed, 1, E)[0] * np.float32(0.05)
    qgu, sgu, qdn, sdn = build_experts(seed, E, H, I, group)
    shared_h = None
    shared_d = None
    if Is:
        a, b = oracle.quantize_w4a16(synth.weights(seed, 2 * Is, H, sub=2 * E), group)
        c, d = oracle.quantize_w4a16(synth.weights(seed, H, Is, sub=2 * E + 1), group)
        shared_h = (a, b, c, d)
        shared_d = tuple(to_dev(v) for v in shared_h)
    xd = xt.cuda()
    y, ids, rw = w4.w4a16_moe_block(xd, to_dev(wr), topk, to_dev(qgu), to_dev(sgu), to_dev(qdn),
                                    to_dev(sdn), shared=shared_d, bias=to_dev(bias),
                                    route_scale=1.5, group=group)
    torch.cuda.synchronize()
    assert w4.w4a16_last_device_status() == w4.W4A16_OK
    # the block routes exactly as the router entry point does
    logits2, ids2, rw2 = w4.w4a16_moe_route(xd, to_dev(wr), topk, bias=to_dev(bias), route_scale=1.5)
    assert torch.equal(ids, ids2) and torch.equal(rw.view(torch.int32), rw2.view(torch.int32))
    ids_h, rw_h = ids.cpu().numpy(), rw.cpu().numpy()
    check_route(logits2.cpu().numpy(), ids_h, rw_h, xt.float().numpy(), wr, bias, topk, 1.5)
    bf16 = dt == "bf16"
    ref, tol = oracle.moe_block_ref(xt.float().numpy(), ids_h, rw_h, qgu, sgu, qdn, sdn, shared_h,
                                    bf16, eps=4e-3 if bf16 else 1e-5, group=group)
    err = np.abs(y.cpu().numpy().astype(np.float64) - ref)
    assert np.all(err <= tol), f"max err/tol = {np.max(err / tol):.3e}"


def test_block_deterministic(w4):
    T, H, I, Is, E, topk = 24, 512, 256, 256, 10, 3
    x = to_dev(synth.activations(9, T, H), torch.bfloat16)
    wr = to_dev(synth.weights(9, E, H, sub=100))
    qgu, sgu, qdn, sdn = (to_dev(v) for v in build_experts(9, E, H, I, 32))
    a, b = oracle.quantize_w4a16(synth.weights(9, 2 * Is, H, sub=2 * E))
    c, d = oracle.quantize_w4a16(synth.weights(9, H, Is, sub=2 * E + 1))
    sh = tuple(to_dev(v) for v in (a, b, c, d))
    y1, _, _ = w4.w4a16_moe_block(x, wr, topk, qgu, sgu, qdn, sdn, shared=sh)
    y2, _, _ = w4.w4a16_moe_block(x, wr, topk, qgu, sgu, qdn, sdn, shared=sh)
    assert torch.equal(y1.view(torch.int32), y2.view(torch.int32))


def test_full_size_block_sampled_tokens(w4):
    T, H, I, Is, E, topk = 128, 7168, 2048, 2048, 384, 8
    seed = 0
    dev = torch.device("cuda")
    x = synth.activations(seed, T, H)
    xb = torch.from_numpy(x).to(torch.bfloat16)
    wr = synth.weights_device(seed + 1, E, H, dev)
    bias = synth.activations(seed + 1, 1, E)[0] * np.float32(0.05)
    qgu = torch.empty((E, 2 * I, H // 8), dtype=torch.int32, device=dev)
    sgu = torch.empty((E, 2 * I, H // 32), dtype=torch.float32, device=dev)
    qdn = torch.empty((E, H, I // 8), dtype=torch.int32, device=dev)
    sdn = torch.empty((E, H, I // 32), dtype=torch.float32, device=dev)
    for e in range(E):
        w4.w4a16_quantize(synth.weights_device(seed, 2 * I, H, dev, sub=2 * e), qw=qgu[e], sc=sgu[e])
        w4.w4a16_quantize(synth.weights_device(seed, H, I, dev, sub=2 * e + 1), qw=qdn[e], sc=sdn[e])
    wsg = synth.weights_device(seed, 2 * Is, H, dev, sub=2 * E)
    wsd = synth.weights_device(seed, H, Is, dev, sub=2 * E + 1)
    sh = w4.w4a16_quantize(wsg) + w4.w4a16_quantize(wsd)
    y, ids, rw = w4.w4a16_moe_block(xb.cuda(), wr, topk, qgu, sgu, qdn, sdn, shared=sh,
                                    bias=to_dev(bias), route_scale=2.827)
    torch.cuda.synchronize()
    assert w4.w4a16_last_device_status() == w4.W4A16_OK
    ids_h, rw_h = ids.cpu().numpy(), rw.cpu().numpy()
    logits, _, _ = w4.w4a16_moe_route(xb.cuda(), wr, topk, bias=to_dev(bias), route_scale=2.827)
    check_route(logits.cpu().numpy(), ids_h, rw_h, xb.float().numpy(), wr.cpu().numpy(), bias,
                topk, 2.827)
    tokens = [0, 77]
    used = sorted({int(e) for t in tokens for e in ids_h[t]})
    hq = {}
    for e in used:
        a, b = oracle.quantize_w4a16(synth.weights_device(seed, 2 * I, H, dev, sub=2 * e).cpu().numpy())
        c, d = oracle.quantize_w4a16(synth.weights_device(seed, H, I, dev, sub=2 * e + 1).cpu().numpy())
        hq[e] = (a, b, c, d)
    shared_h = oracle.quantize_w4a16(wsg.cpu().numpy()) + oracle.quantize_w4a16(wsd.cpu().numpy())
    assert np.array_equal(shared_h[0], sh[0].cpu().numpy())
    ref, tol = oracle.moe_block_ref(xb.float().numpy(), ids_h, rw_h,
                                    {e: v[0] for e, v in hq.items()}, {e: v[1] for e, v in hq.items()},
                                    {e: v[2] for e, v in hq.items()}, {e: v[3] for e, v in hq.items()},
                                    shared_h, True, eps=4e-3, tokens=tokens)
    yh = y.cpu().numpy().astype(np.float64)
    for t in tokens:
        err = np.abs(yh[t] - ref[t])
        assert np.all(err <= tol[t]), f"token {t}: max err/tol = {np.max(err / tol[t]):.3e}"
