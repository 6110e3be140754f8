"""Pins of the CPU oracle against things other than itself.

Each check ties one oracle function to a hand-derived fixture, a closed form,
a brute-force pure-Python loop written independently here, a library routine
or an invariant, chosen so that a plausible slip (nibble order, zero point,
group indexing, a transposed operand, rounding mode, a dropped term) fails.

Format and method: "The Quiet Commit: How a Single Documentation Edit Marks
the Completion of a Major Engineering Milestone", sections "The INT4
Milestone" and "Input Knowledge Required"; "The Silence of Success: A Single
Line That Speaks Volumes", section "What the Edit Actually Built".
"""

import math
import os
import struct
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth


# ------------------------------------------------------------ helpers (independent)
def f32(v: float) -> float:
    """Round a Python float to the nearest fp32 (struct does IEEE RNE)."""
    return struct.unpack("<f", struct.pack("<f", v))[0]


def word_nibble(word: int, j: int) -> int:
    """Nibble j of a 32-bit word given as a Python int (any sign)."""
    return (word & 0xFFFFFFFF) >> (4 * j) & 0xF


def brute_dequant(qw, sc, group=32):
    """Python-int unpacking, one element at a time -> nested lists of floats."""
    N, W = qw.shape
    K = W * 8
    out = [[0.0] * K for _ in range(N)]
    for n in range(N):
        for k in range(K):
            nib = word_nibble(int(qw[n, k // 8]), k % 8)
            out[n][k] = f32((nib - 8) * float(sc[n, k // group]))
    return out


def load_pack_golden(golden_dir):
    rows = []
    with open(os.path.join(golden_dir, "pack_words.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            rows.append(([int(v) for v in parts[:8]], int(parts[8], 16)))
    return rows


def load_quant_golden(golden_dir):
    cases = []
    with open(os.path.join(golden_dir, "quant_groups.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, scale, ws, qs = [p.strip() for p in line.split("|")]
            w = np.zeros(32, np.float32)
            q = np.zeros(32, np.int64)
            for tok in ws.split():
                c, v = tok.split(":")
                w[int(c)] = np.float32(float(v))
            for tok in qs.split():
                c, v = tok.split(":")
                q[int(c)] = int(v)
            cases.append((name, np.float32(float(scale)), w, q))
    return cases


# ------------------------------------------------------------ pack / unpack
def test_pack_matches_hand_derived_words(golden_dir):
    rows = load_pack_golden(golden_dir)
    assert len(rows) >= 10
    q = np.array([r[0] for r in rows], dtype=np.int64)
    nib = q + 8
    qw = oracle.pack_nibbles(nib.reshape(len(rows), 8))
    got = [int(v) & 0xFFFFFFFF for v in qw[:, 0]]
    assert got == [r[1] for r in rows]
    back = oracle.unpack_nibbles(qw).astype(np.int64) - 8
    np.testing.assert_array_equal(back, q)


def test_every_nibble_at_every_position_roundtrips():
    # 16 values x 8 positions, with the other positions holding a different
    # value so a misplaced shift shows; includes words with the top bit set.
    rows = []
    for pos in range(8):
        for v in range(16):
            row = [(v + 5) % 16] * 8
            row[pos] = v
            rows.append(row)
    nib = np.array(rows, dtype=np.int64)
    qw = oracle.pack_nibbles(nib)
    assert (qw < 0).any(), "some words must be negative as int32"
    for r, row in enumerate(rows):
        word = int(qw[r, 0])
        assert [word_nibble(word, j) for j in range(8)] == row
    np.testing.assert_array_equal(oracle.unpack_nibbles(qw), nib.astype(np.uint8))


def test_pack_random_against_python_ints():
    rng = np.random.default_rng(11)
    nib = rng.integers(0, 16, size=(5, 64))
    qw = oracle.pack_nibbles(nib)
    for n in range(5):
        for w in range(8):
            expect = 0
            for j in range(8):
                expect |= int(nib[n, 8 * w + j]) << (4 * j)
            assert int(qw[n, w]) & 0xFFFFFFFF == expect


# ------------------------------------------------------------ dequantisation
def test_dequant_closed_form_all_nibbles():
    # every nibble value, every position, a distinct scale per group so a
    # wrong group index shows
    rng = np.random.default_rng(3)
    N, K = 4, 128
    nib = np.tile(np.arange(16), (N, K // 16))
    rng.permuted(nib, axis=1, out=nib)
    qw = oracle.pack_nibbles(nib)
    sc = (rng.standard_normal((N, K // 32)).astype(np.float32) * np.float32(0.37))
    sc[0, 0] = np.float32(2.0 ** -126)  # smallest normal
    sc[1, 1] = np.float32(0.0)
    got = oracle.dequantize(qw, sc)
    ref = brute_dequant(qw, sc)
    for n in range(N):
        for k in range(K):
            assert got[n, k] == np.float32(ref[n][k])
            # closed form with an exact rational check
            exact = (int(nib[n, k]) - 8) * Fraction(float(sc[n, k // 32]))
            assert got[n, k] == np.float32(f32(float(exact)))


def test_dequant_zero_point_and_extremes():
    nib = np.array([[0, 8, 15, 7, 9, 1, 14, 8]])
    qw = oracle.pack_nibbles(nib)
    sc = np.full((1, 1), np.float32(0.25), dtype=np.float32)
    # K = 8 with group 8 to keep one scale
    got = oracle.dequantize(qw, sc, group=8)
    assert got.tolist() == [[-2.0, 0.0, 1.75, -0.25, 0.25, -1.75, 1.5, 0.0]]


# ------------------------------------------------------------ quantiser
def test_quantizer_hand_cases(golden_dir):
    cases = load_quant_golden(golden_dir)
    assert {c[0] for c in cases} >= {"ties", "negmax", "zero"}
    w = np.stack([c[2] for c in cases])
    qw, sc = oracle.quantize_w4a16(w)
    q = oracle.unpack_nibbles(qw).astype(np.int64) - 8
    for i, (name, scale, _, qexp) in enumerate(cases):
        assert sc[i, 0] == scale, name
        np.testing.assert_array_equal(q[i], qexp, err_msg=name)


def test_quantizer_roundtrip_bound_and_extremes():
    w = synth.weights(0, 64, 1024)
    w[3, 32:64] = 0.0                       # an all-zero group
    w[5, 0:32] = np.float32(1e-30)          # a tiny constant group
    qw, sc = oracle.quantize_w4a16(w)
    what = oracle.dequantize(qw, sc)
    q = oracle.unpack_nibbles(qw).astype(np.int64) - 8
    s_full = np.repeat(sc, 32, axis=1).astype(np.float64)
    err = np.abs(w.astype(np.float64) - what.astype(np.float64))
    # |w - w_hat| <= s/2, plus the fp32 rounding of w/s and of q*s
    assert np.all(err <= s_full * (0.5 + 2.0 ** -20) + 2.0 ** -149)
    assert q.min() >= -7 and q.max() <= 7  # s = max|w|/7 never reaches -8
    G = w.shape[1] // 32
    wg = w.reshape(64, G, 32)
    qg = q.reshape(64, G, 32)
    for n in range(64):
        for g in range(G):
            if sc[n, g] == 0:
                assert not qg[n, g].any()
                continue
            a = int(np.argmax(np.abs(wg[n, g])))
            assert abs(qg[n, g, a]) == 7
            assert np.sign(qg[n, g, a]) == np.sign(wg[n, g, a])
            # scale is max|w| / 7 as an fp32 division
            assert sc[n, g] == np.float32(f32(float(np.abs(wg[n, g]).max()) / 7.0))
    assert sc[3, 1] == 0 and (q[3, 32:64] == 0).all()


def test_quantizer_groups_are_independent():
    w = synth.weights(1, 4, 256)
    qw, sc = oracle.quantize_w4a16(w)
    w2 = w.copy()
    w2[:, 64:96] *= np.float32(100.0)      # change group 2 only
    qw2, sc2 = oracle.quantize_w4a16(w2)
    keep = np.ones(8, bool)
    keep[2] = False
    np.testing.assert_array_equal(sc[:, keep], sc2[:, keep])
    np.testing.assert_array_equal(qw[:, :8], qw2[:, :8])
    np.testing.assert_array_equal(qw[:, 12:], qw2[:, 12:])


def brute_quantize(w, group):
    """Scalar quantiser on Python numbers, one group at a time -> (nibbles, scales).

    s = fp32(max|w| / 7) (a double quotient rounded once more to fp32 is the
    correctly rounded fp32 quotient), q = round-half-even(fp32(w / s))
    clamped to [-8, 7], q = 0 where s = 0."""
    N, K = w.shape
    nib = [[0] * K for _ in range(N)]
    scales = [[0.0] * (K // group) for _ in range(N)]
    for n in range(N):
        for g in range(K // group):
            vals = [float(w[n, g * group + j]) for j in range(group)]
            s = f32(max(abs(v) for v in vals) / 7.0)
            scales[n][g] = s
            for j, v in enumerate(vals):
                q = 0 if s == 0.0 else max(-8, min(7, round(f32(v / s))))
                nib[n][g * group + j] = q + 8
    return nib, scales


@pytest.mark.parametrize("group", [32, 64, 128])
def test_quantizer_against_scalar_loop_all_group_sizes(group):
    N, K = 3, 384
    w = synth.weights(11, N, K)
    w[1, group:2 * group] = 0.0                       # an all-zero group
    w[2, 5] = np.float32(40.0)                        # one outlier sets its group's scale
    qw, sc = oracle.quantize_w4a16(w, group)
    assert qw.shape == (N, K // 8) and sc.shape == (N, K // group)
    nib, scales = brute_quantize(w, group)
    for n in range(N):
        for k in range(K):
            assert word_nibble(int(qw[n, k // 8]), k % 8) == nib[n][k], (n, k)
        for g in range(K // group):
            assert float(sc[n, g]) == scales[n][g], (n, g)
    assert sc[1, 1] == 0.0
    assert sc[2, 0] == np.float32(f32(40.0 / 7.0))
    # a group of 64 or 128 shares one scale where groups of 32 would not
    if group > 32:
        q32, s32 = oracle.quantize_w4a16(w, 32)
        assert not np.array_equal(np.repeat(sc, group // 32, axis=1), s32)


@pytest.mark.parametrize("group", [64, 128])
def test_quantizer_groups_are_independent_larger_groups(group):
    w = synth.weights(12, 4, 512)
    qw, sc = oracle.quantize_w4a16(w, group)
    w2 = w.copy()
    w2[:, group:2 * group] *= np.float32(100.0)       # change group 1 only
    qw2, sc2 = oracle.quantize_w4a16(w2, group)
    keep = np.ones(512 // group, bool)
    keep[1] = False
    np.testing.assert_array_equal(sc[:, keep], sc2[:, keep])
    wpg = group // 8                                  # packed words per group
    np.testing.assert_array_equal(qw[:, :wpg], qw2[:, :wpg])
    np.testing.assert_array_equal(qw[:, 2 * wpg:], qw2[:, 2 * wpg:])
    assert np.all(sc2[:, 1] > 50 * sc[:, 1])           # the changed group's scale follows


def test_dequant_larger_group_uses_one_scale_per_group():
    N, K = 2, 256
    qw = oracle.pack_nibbles(np.tile(np.arange(16, dtype=np.uint8), (N, K // 16)))
    for group in (64, 128):
        sc = (np.arange(N * (K // group), dtype=np.float32).reshape(N, K // group) + 1) * 0.25
        got = oracle.dequantize(qw, sc, group)
        ref = brute_dequant(qw, sc, group)
        np.testing.assert_array_equal(got, np.array(ref, np.float32))
        # column k of row n is (k % 16 - 8) * sc[n][k // group]
        assert got[1, group] == np.float32((group % 16 - 8) * sc[1, 1])


# ------------------------------------------------------------ GEMM
def brute_gemm(x, qw, sc, group=32):
    """Exact rational triple loop: y[m][n] = sum_k x[m][k] * W_hat[n][k]."""
    wd = brute_dequant(qw, sc, group)
    M, K = x.shape
    N = len(wd)
    y = [[Fraction(0)] * N for _ in range(M)]
    b = [[Fraction(0)] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            acb = Fraction(0)
            for k in range(K):
                p = Fraction(float(x[m, k])) * Fraction(wd[n][k])
                acc += p
                acb += abs(p)
            y[m][n] = acc
            b[m][n] = acb
    return y, b


@pytest.mark.parametrize("M,N,K", [(1, 3, 32), (2, 5, 64), (4, 8, 64), (3, 1, 96)])
def test_gemm_matches_exact_triple_loop(M, N, K):
    x = synth.activations(7, M, K)
    w = synth.weights(7, N, K)
    qw, sc = oracle.quantize_w4a16(w)
    y, bound = oracle.gemm_ref(x, qw, sc)
    ye, be = brute_gemm(x, qw, sc)
    for m in range(M):
        for n in range(N):
            # fp64 accumulation of K exact-in-fp64 products
            assert abs(y[m, n] - float(ye[m][n])) <= K * 2.0 ** -52 * float(be[m][n])
            assert bound[m, n] == pytest.approx(float(be[m][n]), rel=1e-13)
    # a transposed operand would not even have this shape
    assert y.shape == (M, N)


@pytest.mark.parametrize("M,N,K,group", [(2, 3, 128, 64), (1, 2, 256, 128), (3, 2, 384, 128)])
def test_gemm_matches_exact_triple_loop_larger_groups(M, N, K, group):
    x = synth.activations(8, M, K)
    w = synth.weights(8, N, K)
    qw, sc = oracle.quantize_w4a16(w, group)
    y, bound = oracle.gemm_ref(x, qw, sc, group)
    ye, be = brute_gemm(x, qw, sc, group)
    for m in range(M):
        for n in range(N):
            assert abs(y[m, n] - float(ye[m][n])) <= K * 2.0 ** -52 * float(be[m][n])
            assert bound[m, n] == pytest.approx(float(be[m][n]), rel=1e-13)


def test_gemm_one_hot_reproduces_columns():
    N, K = 16, 128
    w = synth.weights(5, N, K)
    qw, sc = oracle.quantize_w4a16(w)
    wd = brute_dequant(qw, sc)
    x = np.eye(K, dtype=np.float32)          # row m = e_m
    y, _ = oracle.gemm_ref(x, qw, sc)
    for k in range(K):
        for n in range(N):
            assert y[k, n] == wd[n][k]


def test_gemm_ones_gives_row_sums_and_linearity():
    N, K = 8, 256
    w = synth.weights(9, N, K)
    qw, sc = oracle.quantize_w4a16(w)
    wd = brute_dequant(qw, sc)
    y, b = oracle.gemm_ref(np.ones((1, K), np.float32), qw, sc)
    for n in range(N):
        exact = sum(Fraction(v) for v in wd[n])
        assert abs(y[0, n] - float(exact)) <= 1e-14 * float(b[0, n])
    x1 = synth.activations(1, 2, K)
    x2 = synth.activations(2, 2, K)
    ya, _ = oracle.gemm_ref(x1, qw, sc)
    yb, _ = oracle.gemm_ref(x2, qw, sc)
    yab, bab = oracle.gemm_ref((x1 + x2).astype(np.float32), qw, sc)
    # x1 + x2 rounds in fp32; compare within that rounding
    assert np.all(np.abs(yab - ya - yb) <= 1e-6 * (bab + 1e-30))


def test_gemm_bound_dominates_and_is_tight_for_positive_products():
    K = 64
    nib = np.full((1, K), 15)                # q = 7 everywhere
    qw = oracle.pack_nibbles(nib)
    sc = np.full((1, K // 32), np.float32(0.5))
    x = np.abs(synth.activations(4, 1, K))
    y, b = oracle.gemm_ref(x, qw, sc)
    assert y[0, 0] == pytest.approx(b[0, 0], rel=1e-15)
    assert y[0, 0] == pytest.approx(3.5 * float(x.astype(np.float64).sum()), rel=1e-15)


# ------------------------------------------------------------ bf16 rounding
def test_round_to_bf16_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    a = rng.standard_normal(20000).astype(np.float32) * np.float32(3.0)
    special = np.array([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 1.0078125,
                        65504.0, 3.4e38, 1e-40, -1e-40, np.inf, -np.inf], np.float32)
    # exact ties: low 16 bits = 0x8000 with even and odd bf16 lsb
    ties = np.array([0x3F808000, 0x3F818000, 0xBF808000, 0x40018000], np.uint32).view(np.float32)
    a = np.concatenate([a, special, ties])
    ours = oracle.round_to_bf16(a)
    ref = torch.from_numpy(a).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(ours.view(np.uint32), ref.view(np.uint32))


# ------------------------------------------------------------ MoE pieces
def test_moe_sort_against_brute_force():
    ids, _ = synth.routing(3, 37, 4, 11)
    offsets, perm = oracle.moe_sort(ids, 11)
    flat = [int(v) for v in ids.reshape(-1)]
    expect_perm = []
    expect_off = [0]
    for e in range(11):
        for p, v in enumerate(flat):
            if v == e:
                expect_perm.append(p)
        expect_off.append(len(expect_perm))
    assert perm.tolist() == expect_perm
    assert offsets.tolist() == expect_off


def test_moe_sort_empty_and_single_expert():
    ids = np.zeros((5, 1), np.int32)
    off, perm = oracle.moe_sort(ids, 3)
    assert off.tolist() == [0, 5, 5, 5] and perm.tolist() == [0, 1, 2, 3, 4]
    off, perm = oracle.moe_sort(np.zeros((0, 2), np.int32), 4)
    assert off.tolist() == [0, 0, 0, 0, 0] and perm.tolist() == []
    with pytest.raises(ValueError):
        oracle.moe_sort(np.array([[4]]), 4)


def test_silu_closed_forms():
    g = np.array([0.0, 1.0, -1.0, 30.0, -30.0, 2.5])
    s = oracle.silu(g)
    assert s[0] == 0.0
    assert s[1] == pytest.approx(1.0 / (1.0 + math.exp(-1.0)), rel=1e-15)
    assert s[3] == pytest.approx(30.0, rel=1e-12)
    assert abs(s[4]) < 1e-11
    # silu(g) - silu(-g) = g
    h = np.linspace(-8, 8, 33)
    np.testing.assert_allclose(oracle.silu(h) - oracle.silu(-h), h, rtol=0, atol=1e-14)


def brute_moe(x, ids, rw, qgu, sgu, qdn, sdn, bf16_mode):
    """Pure-Python MoE: loops over tokens, slots, rows and columns."""
    import torch
    T, H = x.shape
    topk = ids.shape[1]
    y = [[0.0] * H for _ in range(T)]
    for t in range(T):
        for j in range(topk):
            e = int(ids[t, j])
            wgu = brute_dequant(qgu[e], sgu[e])
            wdn = brute_dequant(qdn[e], sdn[e])
            I = len(wgu) // 2
            gu = [math.fsum(float(x[t, k]) * wgu[r][k] for k in range(H)) for r in range(2 * I)]
            h = [gu[i] / (1.0 + math.exp(-gu[i])) * gu[I + i] for i in range(I)]
            if bf16_mode:
                h = torch.tensor(h, dtype=torch.float32).to(torch.bfloat16).double().tolist()
            for n in range(H):
                o = math.fsum(h[i] * wdn[n][i] for i in range(I))
                y[t][n] += float(rw[t, j]) * o
    return np.array(y)


def _tiny_moe(seed, T=3, H=32, I=32, E=4, topk=2):
    x = synth.activations(seed, T, H)
    ids, rw = synth.routing(seed, T, topk, E)
    qgu, sgu, qdn, sdn = [], [], [], []
    for e in range(E):
        a, b = oracle.quantize_w4a16(synth.weights(seed, 2 * I, H, sub=2 * e))
        c, d = oracle.quantize_w4a16(synth.weights(seed, H, I, sub=2 * e + 1))
        qgu.append(a); sgu.append(b); qdn.append(c); sdn.append(d)
    return x, ids, rw, np.stack(qgu), np.stack(sgu), np.stack(qdn), np.stack(sdn)


@pytest.mark.parametrize("bf16_mode", [False, True])
def test_moe_ref_matches_brute_force(bf16_mode):
    pytest.importorskip("torch")
    x, ids, rw, qgu, sgu, qdn, sdn = _tiny_moe(21)
    if bf16_mode:
        x = oracle.round_to_bf16(x)
    y, tol = oracle.moe_ref(x, ids, rw, qgu, sgu, qdn, sdn, bf16_mode, eps=4e-3)
    yb = brute_moe(x, ids, rw, qgu, sgu, qdn, sdn, bf16_mode)
    scale = np.abs(yb).max()
    np.testing.assert_allclose(y, yb, rtol=0, atol=1e-12 * scale)
    assert (tol > 0).all() and np.all(tol < 0.5 * np.abs(yb).sum(axis=1, keepdims=True))


def test_moe_ref_top1_unit_weight_is_two_gemms_and_swiglu():
    x, ids, rw, qgu, sgu, qdn, sdn = _tiny_moe(5, T=4, E=3, topk=1)
    rw = np.ones_like(rw)
    y, _ = oracle.moe_ref(x, ids, rw, qgu, sgu, qdn, sdn, False, eps=1e-5)
    for t in range(4):
        e = int(ids[t, 0])
        wgu = np.array(brute_dequant(qgu[e], sgu[e]))
        wdn = np.array(brute_dequant(qdn[e], sdn[e]))
        gu = wgu @ x[t].astype(np.float64)
        g, u = gu[:32], gu[32:]
        h = g * u / (1.0 + np.exp(-g))
        np.testing.assert_allclose(y[t], wdn @ h, rtol=1e-12, atol=1e-14)


def test_moe_ref_token_permutation_and_slot_order():
    x, ids, rw, qgu, sgu, qdn, sdn = _tiny_moe(8, T=5, E=6, topk=3)
    y, _ = oracle.moe_ref(x, ids, rw, qgu, sgu, qdn, sdn, False, eps=1e-5)
    p = np.array([3, 0, 4, 1, 2])
    yp, _ = oracle.moe_ref(x[p], ids[p], rw[p], qgu, sgu, qdn, sdn, False, eps=1e-5)
    np.testing.assert_array_equal(yp, y[p])
    s = np.array([2, 0, 1])
    ys, _ = oracle.moe_ref(x, ids[:, s], rw[:, s], qgu, sgu, qdn, sdn, False, eps=1e-5)
    np.testing.assert_allclose(ys, y, rtol=1e-13, atol=1e-15)
    sub, _ = oracle.moe_ref(x, ids, rw, qgu, sgu, qdn, sdn, False, eps=1e-5, tokens=[1, 3])
    np.testing.assert_array_equal(sub[[1, 3]], y[[1, 3]])
    assert not sub[[0, 2, 4]].any()


def test_moe_swiglu_stage_matches_brute_force():
    """One expert's gate/up GEMM and SwiGLU against a pure-Python loop (exact
    sums with math.fsum), in both modes; the bf16-mode tolerance covers the
    rounding of h to bf16."""
    pytest.importorskip("torch")
    x, ids, rw, qgu, sgu, qdn, sdn = _tiny_moe(31, T=3, E=2)
    for bf16_mode in (False, True):
        xs = oracle.round_to_bf16(x) if bf16_mode else x
        h, tol = oracle.moe_swiglu_ref(xs, qgu[1], sgu[1], bf16_mode, eps=4e-3)
        wgu = brute_dequant(qgu[1], sgu[1])
        I = len(wgu) // 2
        for m in range(xs.shape[0]):
            gu = [math.fsum(float(xs[m, k]) * wgu[r][k] for k in range(xs.shape[1]))
                  for r in range(2 * I)]
            hb = [gu[i] / (1.0 + math.exp(-gu[i])) * gu[I + i] for i in range(I)]
            np.testing.assert_allclose(h[m], hb, rtol=1e-12, atol=1e-15)
        assert (tol > 0).all()
        if bf16_mode:  # the device stores h rounded to bf16
            hb16 = oracle.round_to_bf16(h.astype(np.float32)).astype(np.float64)
            assert np.all(np.abs(hb16 - h) <= tol)


def test_moe_down_stage_matches_brute_force_and_scales():
    """One expert's down GEMM fed a given h, times the routing weight, against
    a pure-Python loop; doubling the weight doubles the output exactly."""
    x, ids, rw, qgu, sgu, qdn, sdn = _tiny_moe(32, T=3, E=2)
    h = synth.activations(33, 3, 32).astype(np.float64)
    r = np.array([0.25, -1.5, 3.0], np.float32)
    o, tol = oracle.moe_down_ref(h, r, qdn[0], sdn[0], eps=4e-3)
    wdn = brute_dequant(qdn[0], sdn[0])
    for m in range(3):
        for n in range(len(wdn)):
            ob = float(r[m]) * math.fsum(h[m, i] * wdn[n][i] for i in range(h.shape[1]))
            assert o[m, n] == pytest.approx(ob, rel=1e-12, abs=1e-15)
    o2, tol2 = oracle.moe_down_ref(h, 2 * r, qdn[0], sdn[0], eps=4e-3)
    np.testing.assert_array_equal(o2, 2 * o)
    np.testing.assert_array_equal(tol2, 2 * tol)
    assert np.all(tol >= 4e-3 * np.abs(o))  # sum|h*w| bounds |sum h*w|


def test_moe_stages_compose_to_the_layer():
    """Top-1 routing in fp32 mode: the layer is the down stage fed the SwiGLU
    stage's h, with the routing weight."""
    x, ids, rw, qgu, sgu, qdn, sdn = _tiny_moe(34, T=4, E=3, topk=1)
    y, _ = oracle.moe_ref(x, ids, rw, qgu, sgu, qdn, sdn, False, eps=1e-5)
    for t in range(4):
        e = int(ids[t, 0])
        h, _ = oracle.moe_swiglu_ref(x[t:t + 1], qgu[e], sgu[e], False, eps=1e-5)
        o, _ = oracle.moe_down_ref(h, rw[t:t + 1, 0], qdn[e], sdn[e], eps=1e-5)
        np.testing.assert_allclose(y[t], o[0], rtol=1e-13, atol=1e-15)


# ------------------------------------------------------------ MoE routing and block
def brute_route(x, wr, bias, topk, scale):
    """Pure-Python routing: exact rational logits, math.exp sigmoid, sort by key."""
    T, H = x.shape
    E = wr.shape[0]
    logits, ids, ws = [], [], []
    for t in range(T):
        lt = [float(sum(Fraction(float(x[t, h])) * Fraction(float(wr[e, h])) for h in range(H)))
              for e in range(E)]
        s = [1.0 / (1.0 + math.exp(-v)) for v in lt]
        b = [0.0] * E if bias is None else [float(v) for v in bias]
        order = sorted(range(E), key=lambda e: (-(s[e] + b[e]), e))[:topk]
        tot = math.fsum(s[e] for e in order)
        logits.append(lt)
        ids.append(order)
        ws.append([scale * s[e] / tot for e in order])
    return logits, ids, ws


@pytest.mark.parametrize("T,E,H,topk,use_bias", [(4, 7, 16, 3, False), (3, 12, 32, 5, True),
                                                 (2, 5, 8, 5, False)])
def test_route_against_brute_force(T, E, H, topk, use_bias):
    x = synth.activations(21, T, H)
    wr = synth.weights(21, E, H)
    bias = (synth.weights(22, 1, E)[0] * np.float32(0.1)) if use_bias else None
    logits, bound, ids, w = oracle.moe_route_ref(x, wr, bias, topk, 2.5)
    bl, bi, bw = brute_route(x, wr, bias, topk, 2.5)
    np.testing.assert_array_equal(ids, np.array(bi))
    np.testing.assert_allclose(logits, np.array(bl), rtol=0, atol=1e-12)
    np.testing.assert_allclose(w, np.array(bw), rtol=1e-13, atol=0)
    assert np.all(bound >= np.abs(logits))
    np.testing.assert_allclose(w.sum(axis=1), 2.5, rtol=1e-14)      # weights sum to the scale


def test_route_ties_bias_and_full_selection():
    H = 8
    x = np.ones((1, H), np.float32)
    wr = np.zeros((6, H), np.float32)
    wr[1] = wr[4] = 0.25                      # experts 1 and 4: equal logits 2.0
    wr[2] = -0.5                              # expert 2: logit -4
    _, _, ids, w = oracle.moe_route_ref(x, wr, None, 2, 1.0)
    assert list(ids[0]) == [1, 4]             # the tie goes to the lower id first
    np.testing.assert_allclose(w[0], [0.5, 0.5], rtol=1e-15)
    # a large bias forces expert 2 in; its weight still uses the plain sigmoid
    bias = np.zeros(6, np.float32)
    bias[2] = 10.0
    _, _, ids, w = oracle.moe_route_ref(x, wr, bias, 2, 1.0)
    assert list(ids[0]) == [2, 1]
    s2, s1 = 1 / (1 + math.exp(4.0)), 1 / (1 + math.exp(-2.0))
    np.testing.assert_allclose(w[0], [s2 / (s1 + s2), s1 / (s1 + s2)], rtol=1e-14)
    # topk = E: every expert, in decreasing score order, ties by id
    _, _, ids, w = oracle.moe_route_ref(x, wr, None, 6, 3.0)
    assert list(ids[0]) == [1, 4, 0, 3, 5, 2]
    s = np.array([0.5, s1, s2, 0.5, s1, 0.5])
    np.testing.assert_allclose(w[0], 3.0 * s[[1, 4, 0, 3, 5, 2]] / s.sum(), rtol=1e-14)


def _small_experts(seed, E, H, I, group=32):
    out = [[], [], [], []]
    for e in range(E):
        a, b = oracle.quantize_w4a16(synth.weights(seed, 2 * I, H, sub=2 * e), group)
        c, d = oracle.quantize_w4a16(synth.weights(seed, H, I, sub=2 * e + 1), group)
        for lst, v in zip(out, (a, b, c, d)):
            lst.append(v)
    return [np.stack(v) for v in out]


def test_moe_block_shared_expert_closed_forms():
    T, H, I, Is, E, topk = 3, 64, 32, 64, 4, 2
    x = synth.activations(31, T, H)
    ids, rw = synth.routing(31, T, topk, E)
    qgu, sgu, qdn, sdn = _small_experts(31, E, H, I)
    a, b = oracle.quantize_w4a16(synth.weights(32, 2 * Is, H))
    c, d = oracle.quantize_w4a16(synth.weights(33, H, Is))
    shared = (a, b, c, d)
    base, _ = oracle.moe_ref(x, ids, rw, qgu, sgu, qdn, sdn, False, 1e-5)
    # no shared expert: the routed layer
    y0, _ = oracle.moe_block_ref(x, ids, rw, qgu, sgu, qdn, sdn, None, False, 1e-5)
    np.testing.assert_array_equal(y0, base)
    # a shared expert with all-zero scales adds nothing
    y1, _ = oracle.moe_block_ref(x, ids, rw, qgu, sgu, qdn, sdn,
                                 (a, np.zeros_like(b), c, np.zeros_like(d)), False, 1e-5)
    np.testing.assert_allclose(y1, base, rtol=0, atol=1e-15)
    # routing weights all zero: the shared expert alone, i.e. two GEMMs and SwiGLU
    y2, tol2 = oracle.moe_block_ref(x, ids, np.zeros_like(rw), qgu, sgu, qdn, sdn, shared,
                                    False, 1e-5)
    gu, _ = oracle.gemm_ref(x, a, b)
    h = oracle.silu(gu[:, :Is]) * gu[:, Is:]
    yd = h @ oracle.dequantize(c, d).astype(np.float64).T   # h kept in fp64, as in fp32 mode
    np.testing.assert_allclose(y2, yd, rtol=1e-12, atol=1e-14)
    assert np.all(tol2 > 0)
    # linearity in the routed part: block = routed layer + shared alone
    y3, _ = oracle.moe_block_ref(x, ids, rw, qgu, sgu, qdn, sdn, shared, False, 1e-5)
    np.testing.assert_allclose(y3, base + y2, rtol=1e-12, atol=1e-12)


def test_moe_block_bf16_mode_is_routed_layer_plus_shared_expert():
    """In bf16 mode each expert rounds its own h to bf16, so the block is still
    the routed layer plus the shared expert alone (run as a top-1 layer with
    unit weight), and the bound adds up the same way."""
    T, H, I, Is, E, topk = 4, 64, 32, 64, 5, 3
    x = oracle.round_to_bf16(synth.activations(41, T, H))
    ids, rw = synth.routing(41, T, topk, E)
    qgu, sgu, qdn, sdn = _small_experts(41, E, H, I)
    a, b = oracle.quantize_w4a16(synth.weights(42, 2 * Is, H))
    c, d = oracle.quantize_w4a16(synth.weights(43, H, Is))
    yb, tb = oracle.moe_block_ref(x, ids, rw, qgu, sgu, qdn, sdn, (a, b, c, d), True, 4e-3)
    yr, tr = oracle.moe_ref(x, ids, rw, qgu, sgu, qdn, sdn, True, 4e-3)
    ys, ts = oracle.moe_ref(x, np.zeros((T, 1), np.int32), np.ones((T, 1), np.float32),
                            a[None], b[None], c[None], d[None], True, 4e-3)
    np.testing.assert_allclose(yb, yr + ys, rtol=1e-12, atol=1e-12)
    # the block's bound covers both parts (slot-sum term grows by one slot)
    assert np.all(tb >= tr + ts - 1e-12 * (np.abs(yr) + np.abs(ys)))
