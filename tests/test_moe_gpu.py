"""Parity of the CUDA grouped MoE path with the CPU oracle, through the C ABI.

* the expert sort (offsets, perm) is bit-exact against the oracle's stable
  sort, including ids shared by many tokens, unused experts and E = 1;
* small MoE layers in fp32 and bf16 modes match moe_ref within its
  propagated bound (each GEMM within 1e-5 / 4e-3 of sum|a*w|, through
  SwiGLU, the bf16 rounding of h and the slot sum);
* the full-size layer (128 tokens, hidden 7168, 384 experts of 2048-wide
  SwiGLU, top-8) is checked on sampled tokens: the oracle rebuilds the
  experts those tokens use from the same seeded draws;
* stage by stage (the device leaves its intermediates in the workspace,
  w4a16_moe_workspace_layout says where): the expert-sorted pair order is
  bit-exact; each SwiGLU output h is within the gate/up GEMM bound
  propagated through SwiGLU (plus the bf16 rounding of h in bf16 mode);
  each per-slot output o is within the down GEMM's own bound when the
  oracle's down GEMM is fed the device's h; y is the slot-ordered fp32 sum
  of the device's o. At full size the stage checks cover every token of
  experts chosen to have 1, 2, 3 and more than 3 tokens.
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


@pytest.mark.parametrize("T,topk,E", [(128, 8, 384), (37, 4, 11), (300, 1, 1), (1, 1, 5),
                                      (1000, 8, 64), (64, 6, 8192)])
def test_sort_bit_exact(w4, T, topk, E):
    ids, _ = synth.routing(T + E, T, topk, E)
    off, perm = w4.w4a16_moe_sort(torch.from_numpy(ids).cuda(), E)
    ro, rp = oracle.moe_sort(ids, E)
    np.testing.assert_array_equal(off.cpu().numpy(), ro)
    np.testing.assert_array_equal(perm.cpu().numpy(), rp)
    assert w4.w4a16_last_device_status() == w4.W4A16_OK


def test_sort_skewed_and_invalid(w4):
    ids = np.zeros((50, 4), np.int32)
    ids[:, 1] = 3
    ids[7, 2] = 2
    off, perm = w4.w4a16_moe_sort(torch.from_numpy(ids).cuda(), 4)
    ro, rp = oracle.moe_sort(ids, 4)
    np.testing.assert_array_equal(off.cpu().numpy(), ro)
    np.testing.assert_array_equal(perm.cpu().numpy(), rp)
    # an id out of range is reported through the device status word
    bad = ids.copy()
    bad[3, 0] = 9
    w4.w4a16_moe_sort(torch.from_numpy(bad).cuda(), 4)
    assert w4.w4a16_last_device_status() == w4.W4A16_ERR_INVALID_ARG
    assert w4.w4a16_last_device_status() == w4.W4A16_OK  # cleared by the read


def build_experts_host(seed, E, H, I, group=32):
    qgu, sgu, qdn, sdn = [], [], [], []
    for e in range(E):
        a, b = oracle.quantize_w4a16(synth.weights(seed, 2 * I, H, sub=2 * e), group)
        c, d = oracle.quantize_w4a16(synth.weights(seed, H, I, sub=2 * e + 1), group)
        qgu.append(a); sgu.append(b); qdn.append(c); sdn.append(d)
    return np.stack(qgu), np.stack(sgu), np.stack(qdn), np.stack(sdn)


def read_stages(w4, ws, T, topk, E, H, I, bf16):
    """The device's intermediates from the workspace: perm [n], h [n, I]
    (by sorted position, as float64) and o [n, H] (by pair)."""
    L = w4.w4a16_moe_workspace_layout(T, topk, E, H, I)
    n = T * topk
    raw = ws.cpu()
    perm = raw[L["perm"]:L["perm"] + 4 * n].view(torch.int32).numpy().copy()
    hb = raw[L["h"]:L["h"] + (2 if bf16 else 4) * n * I]
    h = (hb.view(torch.bfloat16).float() if bf16 else hb.view(torch.float32)).numpy()
    o = raw[L["o"]:L["o"] + 4 * n * H].view(torch.float32).numpy()
    return perm, h.reshape(n, I).astype(np.float64), o.reshape(n, H).astype(np.float64)


def check_stages(x, ids, rw, experts, perm, h, o, y, bf16, eps, group=32, only=None):
    """Stage-wise parity. `experts[e]` = (qw_gu, sc_gu, qw_dn, sc_dn) host
    arrays; `only` restricts the h and o checks to those experts."""
    T, topk = ids.shape
    _, ro = oracle.moe_sort(ids, max(int(ids.max()) + 1, 1))
    np.testing.assert_array_equal(perm, ro)
    pos = {int(p): s for s, p in enumerate(perm)}
    by_expert = {}
    for p in range(T * topk):
        by_expert.setdefault(int(ids.reshape(-1)[p]), []).append(p)
    checked = 0
    for e, pairs in sorted(by_expert.items()):
        if only is not None and e not in only:
            continue
        qgu, sgu, qdn, sdn = experts[e]
        toks = [p // topk for p in pairs]
        hr, ht = oracle.moe_swiglu_ref(x[toks], qgu, sgu, bf16, eps, group)
        hd = h[[pos[p] for p in pairs]]
        err = np.abs(hd - hr)
        assert np.all(err <= ht), f"expert {e} h: max err/tol {np.max(err / ht):.3e}"
        rws = rw.reshape(-1)[pairs]
        orf, ot = oracle.moe_down_ref(hd, rws, qdn, sdn, eps, group)
        err = np.abs(o[pairs] - orf)
        assert np.all(err <= ot), f"expert {e} o: max err/tol {np.max(err / ot):.3e}"
        checked += len(pairs)
    # combine: y[t] is the fp32 sum of the token's slots in slot order
    os_ = o.reshape(T, topk, -1)
    ysum = os_.sum(axis=1)
    bound = topk * 2.0 ** -24 * np.abs(os_).sum(axis=1)
    assert np.all(np.abs(y - ysum) <= bound)
    return checked


def check_moe(w4, x, ids, rw, qgu, sgu, qdn, sdn, bf16, group=32):
    xt = torch.from_numpy(x)
    if bf16:
        xt = xt.to(torch.bfloat16)
    dev = [torch.from_numpy(a).cuda() for a in (qgu, sgu, qdn, sdn)]
    T, H = x.shape
    topk, E, I = ids.shape[1], qgu.shape[0], qgu.shape[1] // 2
    ws = torch.empty(w4.w4a16_moe_workspace_size(T, topk, E, H, I), dtype=torch.uint8,
                     device="cuda")
    y = w4.w4a16_moe_gemm(xt.cuda(), torch.from_numpy(ids).cuda(), torch.from_numpy(rw).cuda(),
                          *dev, workspace=ws, group=group)
    torch.cuda.synchronize()
    assert w4.w4a16_last_device_status() == w4.W4A16_OK
    eps = 4e-3 if bf16 else 1e-5
    xo = xt.float().numpy()
    ref, tol = oracle.moe_ref(xo, ids, rw, qgu, sgu, qdn, sdn, bf16, eps=eps, group=group)
    yh = y.cpu().numpy().astype(np.float64)
    err = np.abs(yh - ref)
    assert np.all(err <= tol), f"max err/tol = {np.max(err / tol):.3e}"
    perm, h, o = read_stages(w4, ws, T, topk, E, H, I, bf16)
    experts = {e: (qgu[e], sgu[e], qdn[e], sdn[e]) for e in range(E)}
    check_stages(xo, ids, rw, experts, perm, h, o, yh, bf16, eps, group)
    return y


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("T,H,I,E,topk", [(5, 256, 128, 6, 2), (16, 1024, 512, 9, 4),
                                          (3, 160, 96, 3, 3), (40, 512, 256, 4, 1)])
def test_small_moe(w4, bf16, T, H, I, E, topk):
    seed = T + H + E
    x = synth.activations(seed, T, H)
    ids, rw = synth.routing(seed, T, topk, E)
    qgu, sgu, qdn, sdn = build_experts_host(seed, E, H, I)
    check_moe(w4, x, ids, rw, qgu, sgu, qdn, sdn, bf16)


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("group", [64, 128])
@pytest.mark.parametrize("T,H,I,E,topk", [(5, 256, 128, 6, 2), (16, 1024, 384, 9, 4),
                                          (16, 1024, 512, 9, 4), (100, 768, 512, 5, 3)])
def test_small_moe_group_sizes(w4, bf16, group, T, H, I, E, topk):
    """Groups of 64 and 128 on both expert GEMMs; I = 384 with group 128
    gives 3 scales per down-projection row (loaded per lane, not staged).
    The last two shapes take the tensor-core expert GEMMs in bf16 mode
    (H and I multiples of 256, at least 16 pairs); the last gives experts
    several 16-token tiles with a ragged final one."""
    seed = T + H + E + group
    x = synth.activations(seed, T, H)
    ids, rw = synth.routing(seed, T, topk, E)
    qgu, sgu, qdn, sdn = build_experts_host(seed, E, H, I, group)
    check_moe(w4, x, ids, rw, qgu, sgu, qdn, sdn, bf16, group)


@pytest.mark.parametrize("T,topk,E,H,I", [(4, 4, 4, 256, 256), (2, 8, 8, 512, 256)])
def test_moe_tensor_core_path_smallest(w4, T, topk, E, H, I):
    """Exactly 16 (token, slot) pairs (the fewest the tensor-core expert path
    takes) in bf16 mode, H and I at their 256 minimum or just above: every
    expert has a single, partly filled 16-token tile."""
    x = synth.activations(T * 7 + E, T, H)
    ids, rw = synth.routing(T * 7 + E, T, topk, E)
    qgu, sgu, qdn, sdn = build_experts_host(T * 7 + E, E, H, I)
    check_moe(w4, x, ids, rw, qgu, sgu, qdn, sdn, True)


def test_moe_many_tokens_one_expert(w4):
    # every token routed to expert 0 in slot 0: its weights serve 37 tokens
    T, H, I, E, topk = 37, 512, 256, 3, 2
    x = synth.activations(1, T, H)
    ids, rw = synth.routing(1, T, topk, E)
    ids[:, 0] = 0
    ids[:, 1] = np.where(ids[:, 1] == 0, 1, ids[:, 1])
    qgu, sgu, qdn, sdn = build_experts_host(1, E, H, I)
    check_moe(w4, x, ids, rw, qgu, sgu, qdn, sdn, True)


def test_moe_deterministic(w4):
    T, H, I, E, topk = 8, 512, 256, 5, 2
    x = torch.from_numpy(synth.activations(2, T, H)).to(torch.bfloat16).cuda()
    ids, rw = synth.routing(2, T, topk, E)
    dev = [torch.from_numpy(a).cuda() for a in build_experts_host(2, E, H, I)]
    a = w4.w4a16_moe_gemm(x, torch.from_numpy(ids).cuda(), torch.from_numpy(rw).cuda(), *dev)
    b = w4.w4a16_moe_gemm(x, torch.from_numpy(ids).cuda(), torch.from_numpy(rw).cuda(), *dev)
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_full_size_moe_sampled_tokens(w4):
    T, H, I, E, topk = 128, 7168, 2048, 384, 8
    seed = 0
    dev = torch.device("cuda")
    x = synth.activations(seed, T, H)
    ids, rw = synth.routing(seed, T, topk, E)
    qgu = torch.empty((E, 2 * I, H // 8), dtype=torch.int32, device=dev)
    sgu = torch.empty((E, 2 * I, H // 32), dtype=torch.float32, device=dev)
    qdn = torch.empty((E, H, I // 8), dtype=torch.int32, device=dev)
    sdn = torch.empty((E, H, I // 32), dtype=torch.float32, device=dev)
    for e in range(E):
        w4.w4a16_quantize(synth.weights_device(seed, 2 * I, H, dev, sub=2 * e), qw=qgu[e], sc=sgu[e])
        w4.w4a16_quantize(synth.weights_device(seed, H, I, dev, sub=2 * e + 1), qw=qdn[e], sc=sdn[e])
    xb = torch.from_numpy(x).to(torch.bfloat16)
    ws = torch.empty(w4.w4a16_moe_workspace_size(T, topk, E, H, I), dtype=torch.uint8, device=dev)
    y = w4.w4a16_moe_gemm(xb.cuda(), torch.from_numpy(ids).cuda(), torch.from_numpy(rw).cuda(),
                          qgu, sgu, qdn, sdn, workspace=ws)
    torch.cuda.synchronize()
    assert w4.w4a16_last_device_status() == w4.W4A16_OK
    yh = y.cpu().numpy().astype(np.float64)
    xo = xb.float().numpy()

    # experts with 1, 2, 3 and the most tokens (two of each), plus the
    # experts of two sampled tokens for the end-to-end check
    counts = np.bincount(ids.reshape(-1), minlength=E)
    chosen = []
    for c in (1, 2, 3):
        chosen += [int(e) for e in np.flatnonzero(counts == c)[:2]]
    chosen += [int(e) for e in np.argsort(-counts, kind="stable")[:2]]
    assert counts[chosen[-1]] > 3
    tokens = [0, 77]
    used = sorted(set(chosen) | {int(e) for t in tokens for e in ids[t]})
    hq = {}
    for e in used:
        wg = synth.weights_device(seed, 2 * I, H, dev, sub=2 * e).cpu().numpy()
        wd = synth.weights_device(seed, H, I, dev, sub=2 * e + 1).cpu().numpy()
        a, b = oracle.quantize_w4a16(wg)
        c, d = oracle.quantize_w4a16(wd)
        # the device packing the GPU used is the oracle's packing
        assert np.array_equal(a, qgu[e].cpu().numpy()) and np.array_equal(c, qdn[e].cpu().numpy())
        hq[e] = (a, b, c, d)

    perm, h, o = read_stages(w4, ws, T, topk, E, H, I, True)
    checked = check_stages(xo, ids, rw, hq, perm, h, o, yh, True, 4e-3, only=set(chosen))
    covered = {p // topk for p in range(T * topk) if int(ids.reshape(-1)[p]) in chosen}
    assert checked >= 16 and len(covered) >= 16

    ref, tol = oracle.moe_ref(xo, ids, rw,
                              {e: v[0] for e, v in hq.items()}, {e: v[1] for e, v in hq.items()},
                              {e: v[2] for e, v in hq.items()}, {e: v[3] for e, v in hq.items()},
                              True, eps=4e-3, tokens=tokens)
    for t in tokens:
        err = np.abs(yh[t] - ref[t])
        assert np.all(err <= tol[t]), f"token {t}: max err/tol = {np.max(err / tol[t]):.3e}"
