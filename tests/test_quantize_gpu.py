"""The device quantiser is bit-exact against the oracle's quantiser: the
quantised codes are an integer decision taken in the same fp32 arithmetic on
both sides (max|w| / 7 and w / s as IEEE divisions, round half to even)."""

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


def check(w4, w, group=32):
    qw_d, sc_d = w4.w4a16_quantize(torch.from_numpy(w).cuda(), group=group)
    qw_h, sc_h = oracle.quantize_w4a16(w, group)
    np.testing.assert_array_equal(qw_d.cpu().numpy(), qw_h)
    np.testing.assert_array_equal(sc_d.cpu().numpy().view(np.uint32), sc_h.view(np.uint32))


@pytest.mark.parametrize("N,K", [(1, 32), (3, 96), (512, 256), (4096, 7168), (7, 4128)])
def test_quantizer_random(w4, N, K):
    check(w4, synth.weights(N + K, N, K))



def test_quantizer_edge_groups(w4):
    K = 128
    w = np.zeros((6, K), np.float32)
    # exact ties w/s = k + 0.5 (s = 1): round half to even
    w[0, :10] = [7.0, 3.5, -3.5, 2.5, -0.5, 0.5, 1.5, -2.5, 6.5, -6.5]
    # an all-zero group next to a normal one
    w[1, 32:64] = synth.weights(1, 1, 32)[0]
    # a group with one non-zero entry
    w[2, 70] = np.float32(-1e-3)
    # huge and tiny magnitudes
    w[3, :32] = np.float32(3e38) * np.sign(synth.weights(2, 1, 32)[0])
    w[4, :32] = np.float32(1e-38) * synth.weights(3, 1, 32)[0]
    w[5] = synth.weights(4, 1, K)[0]
    check(w4, w)


def test_quantizer_matches_random_mixed_scales(w4):
    w = synth.weights(5, 256, 1024)
    w *= np.float32(10.0) ** np.random.default_rng(0).uniform(-6, 6, size=(256, 1)).astype(np.float32)
    check(w4, w.astype(np.float32))


@pytest.mark.parametrize("group", [64, 128])
@pytest.mark.parametrize("N,K", [(1, 128), (3, 384), (512, 1024), (4096, 7168), (7, 4224)])
def test_quantizer_group_sizes(w4, group, N, K):
    w = synth.weights(N + K + group, N, K)
    w[0, :group] = 0.0                                # an all-zero group
    w[-1, (group + 3) % K] = np.float32(-25.0)        # an outlier owning a group's scale
    check(w4, w, group)
