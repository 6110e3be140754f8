"""Failure detection without a GPU fault: every device-side wait in the
library is bounded. The host-side switch w4a16_debug_fault_next_launch makes
the next launch of a CUDA-core GEMM kernel (decode GEMV or streaming) skip
its weight copies - a signal nothing
will ever deliver - so its waits run out after about a second; the kernel
records W4A16_ERR_TIMEOUT in the status word and returns. The test checks
the status, that the wait really was bounded, and that the context is still
usable (the next call is correct)."""

import time

import numpy as np
import pytest

import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w4():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import int4_w4a16_group_gemm_gb300 as w4
    return w4


@pytest.mark.parametrize("algo", ["gemv", "stream"])
def test_timeout_is_reported_and_context_survives(w4, algo):
    M, N, K = 1, 1024, 2048
    x = torch.from_numpy(synth.activations(21, M, K)).cuda()
    qw, sc = w4.w4a16_quantize(torch.from_numpy(synth.weights(21, N, K)).cuda())
    ref = w4.w4a16_gemm(x, qw, sc, algo=algo)
    assert w4.w4a16_last_device_status() == w4.W4A16_OK

    w4.w4a16_debug_fault_next_launch(True)
    t0 = time.time()
    w4.w4a16_gemm(x, qw, sc, algo=algo)
    status = w4.w4a16_last_device_status()   # synchronises the stream
    elapsed = time.time() - t0
    assert status == w4.W4A16_ERR_TIMEOUT
    assert 0.5 < elapsed < 30.0

    # the switch cleared itself; the context works and results are right
    y = w4.w4a16_gemm(x, qw, sc, algo=algo)
    assert w4.w4a16_last_device_status() == w4.W4A16_OK
    assert torch.equal(y.view(torch.int32), ref.view(torch.int32))
    assert np.isfinite(y.cpu().numpy()).all()
