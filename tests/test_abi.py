"""The C-ABI library loads and exports every entry point include/w4a16.h
declares; host-side argument checks return their status codes without a
GPU (no compute call is made here)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w4a16.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(w4a16_[a-z_0-9]+)\s*\(", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def w4():
    import int4_w4a16_group_gemm_gb300 as w4
    return w4


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["w4a16_gemm", "w4a16_gemm_ex", "w4a16_quantize", "w4a16_moe_sort",
              "w4a16_moe_workspace_size", "w4a16_moe_gemm", "w4a16_status_string",
              "w4a16_last_device_status"]:
        assert n in names


def test_library_exports_every_declared_symbol(w4):
    lib = ctypes.CDLL(w4.LIB_PATH)
    for n in declared_functions():
        assert hasattr(lib, n), f"{n} not exported"
    # the binding wraps every declared function with a signature
    assert set(declared_functions()) <= set(w4.SIGNATURES)


def test_status_strings(w4):
    assert w4.status_string(0) == "W4A16_OK"
    assert w4.status_string(5) == "W4A16_ERR_TIMEOUT"
    assert w4.status_string(6) == "W4A16_ERR_BOUNDS"
    assert w4.status_string(99) == "W4A16_ERR_UNKNOWN"


def test_bounds_checking_build_compiles_and_exports_the_boundary():
    """The W4A16_DEBUG build (kernels check their indices and record
    W4A16_ERR_BOUNDS) compiles from the same sources and exports every
    declared entry point; its GPU test runs the shapes through it."""
    from int4_w4a16_group_gemm_gb300 import build
    path = build.build(debug=True)
    lib = ctypes.CDLL(path)
    for n in declared_functions():
        assert hasattr(lib, n), f"{n} not exported by the checked build"


def test_host_argument_checks_need_no_gpu(w4):
    lib = w4.lib
    null = ctypes.c_void_p(0)
    fake = ctypes.c_void_p(0x1000)       # never dereferenced: checks fail first
    odd = ctypes.c_void_p(0x1004)
    # null pointers
    assert lib.w4a16_gemm(null, 0, fake, fake, 1, 1, 32, 32, fake, null) == w4.W4A16_ERR_INVALID_ARG
    # sizes
    assert lib.w4a16_gemm(fake, 0, fake, fake, 0, 1, 32, 32, fake, null) == w4.W4A16_ERR_INVALID_ARG
    assert lib.w4a16_gemm(fake, 0, fake, fake, 1, 1, 48, 32, fake, null) == w4.W4A16_ERR_INVALID_ARG
    # group sizes: 32, 64 and 128 only; K a multiple of the group
    for g in (16, 48, 256):
        assert lib.w4a16_gemm(fake, 0, fake, fake, 1, 1, 256, g, fake, null) == w4.W4A16_ERR_UNSUPPORTED
    assert lib.w4a16_gemm(fake, 0, fake, fake, 1, 1, 96, 64, fake, null) == w4.W4A16_ERR_INVALID_ARG
    assert lib.w4a16_gemm(fake, 0, fake, fake, 1, 1, 192, 128, fake, null) == w4.W4A16_ERR_INVALID_ARG
    assert lib.w4a16_gemm_launches(1, 64, 192, 64, 0, 0) >= 1
    assert lib.w4a16_gemm_launches(1, 64, 256, 128, 1, 0) >= 1
    # bad activation dtype
    assert lib.w4a16_gemm(fake, 7, fake, fake, 1, 1, 32, 32, fake, null) == w4.W4A16_ERR_INVALID_ARG
    # misaligned operand
    assert lib.w4a16_gemm(odd, 0, fake, fake, 1, 1, 32, 32, fake, null) == w4.W4A16_ERR_ALIGNMENT
    # bad algo
    assert lib.w4a16_gemm_ex(fake, 0, fake, fake, 1, 1, 32, 32, fake, 9, 0, null) == w4.W4A16_ERR_INVALID_ARG
    # unknown launch flag
    assert lib.w4a16_gemm_ex(fake, 0, fake, fake, 1, 1, 32, 32, fake, 0, 4, null) == w4.W4A16_ERR_INVALID_ARG
    # the bf16-output flag is known: the call gets as far as the alignment check
    assert lib.w4a16_gemm_ex(fake, 0, fake, fake, 1, 1, 32, 32, odd, 0, 2, null) == w4.W4A16_ERR_ALIGNMENT
    # quantiser
    assert lib.w4a16_quantize(null, 4, 32, 32, fake, fake, null) == w4.W4A16_ERR_INVALID_ARG
    assert lib.w4a16_quantize(fake, 4, 40, 32, fake, fake, null) == w4.W4A16_ERR_INVALID_ARG
    assert lib.w4a16_quantize(fake, 4, 96, 64, fake, fake, null) == w4.W4A16_ERR_INVALID_ARG
    assert lib.w4a16_quantize(fake, 4, 256, 16, fake, fake, null) == w4.W4A16_ERR_UNSUPPORTED
    # sort
    assert lib.w4a16_moe_sort(fake, 4, 0, fake, fake, null) == w4.W4A16_ERR_INVALID_ARG
    assert lib.w4a16_moe_sort(fake, 4, 9000, fake, fake, null) == w4.W4A16_ERR_UNSUPPORTED
    # MoE: workspace too small
    ws = w4.w4a16_moe_workspace_size(4, 2, 3, 64, 64)
    assert lib.w4a16_moe_gemm(fake, 1, fake, fake, 4, 2, fake, fake, fake, fake, 3, 64, 64, 32,
                              fake, max(ws - 1, 0), fake, null) == w4.W4A16_ERR_INVALID_ARG
    assert lib.w4a16_moe_gemm(fake, 1, fake, fake, 4, 2, fake, fake, fake, fake, 3, 64, 48, 32,
                              fake, ws, fake, null) == w4.W4A16_ERR_INVALID_ARG
    # H = 192 is not a multiple of group 128; group 16 is not taken
    ws = w4.w4a16_moe_workspace_size(4, 2, 3, 192, 128)
    assert lib.w4a16_moe_gemm(fake, 1, fake, fake, 4, 2, fake, fake, fake, fake, 3, 192, 128, 128,
                              fake, ws, fake, null) == w4.W4A16_ERR_INVALID_ARG
    assert lib.w4a16_moe_gemm(fake, 1, fake, fake, 4, 2, fake, fake, fake, fake, 3, 192, 128, 16,
                              fake, ws, fake, null) == w4.W4A16_ERR_UNSUPPORTED


def test_workspace_size_grows_with_tokens(w4):
    a = w4.w4a16_moe_workspace_size(128, 8, 384, 7168, 2048)
    b = w4.w4a16_moe_workspace_size(256, 8, 384, 7168, 2048)
    assert 0 < a < b
    assert w4.w4a16_moe_workspace_size(-1, 8, 384, 7168, 2048) == 0


def test_router_and_block_argument_checks_need_no_gpu(w4):
    lib = w4.lib
    null = ctypes.c_void_p(0)
    fake = ctypes.c_void_p(0x1000)
    odd = ctypes.c_void_p(0x1004)
    f = ctypes.c_float
    route = lambda x, T, H, wr, E, k, scale: lib.w4a16_moe_route(  # noqa: E731
        x, 0, T, H, wr, null, E, k, f(scale), fake, fake, fake, null)
    assert route(null, 4, 64, fake, 8, 2, 1.0) == w4.W4A16_ERR_INVALID_ARG
    assert route(fake, 4, 64, fake, 8, 9, 1.0) == w4.W4A16_ERR_INVALID_ARG      # topk > E
    assert route(fake, 4, 48, fake, 8, 2, 1.0) == w4.W4A16_ERR_INVALID_ARG      # H % 32
    assert route(fake, 4, 64, fake, 8, 2, float("nan")) == w4.W4A16_ERR_INVALID_ARG
    assert route(fake, 4, 64, fake, 2000, 8, 1.0) == w4.W4A16_ERR_UNSUPPORTED   # E > 1024
    assert route(fake, 4, 64, fake, 100, 40, 1.0) == w4.W4A16_ERR_UNSUPPORTED   # topk > 32
    assert route(odd, 4, 64, fake, 8, 2, 1.0) == w4.W4A16_ERR_ALIGNMENT

    # workspace: the grouped layer's, then logits and the shared expert's buffers
    base = w4.w4a16_moe_workspace_size(128, 8, 384, 7168, 2048)
    no_shared = w4.w4a16_moe_block_workspace_size(128, 8, 384, 7168, 2048, 0)
    with_shared = w4.w4a16_moe_block_workspace_size(128, 8, 384, 7168, 2048, 2048)
    assert base + 128 * 384 * 4 <= no_shared < with_shared
    assert with_shared - no_shared >= 128 * (2 * 2048 + 2048 + 7168) * 4
    assert w4.w4a16_moe_block_workspace_size(4, 2, 3, 64, 64, -1) == 0

    def block(Is, sh, group=32, ws=None, H=64, I=64):
        wsz = w4.w4a16_moe_block_workspace_size(4, 2, 3, H, I, max(Is, 0)) if ws is None else ws
        return lib.w4a16_moe_block(fake, 1, 4, fake, null, 3, 2, f(1.0), fake, fake, fake, fake,
                                   H, I, sh, sh, sh, sh, Is, group, fake, wsz, fake, fake, fake,
                                   null)
    assert block(64, null) == w4.W4A16_ERR_INVALID_ARG          # shared width, no weights
    assert block(48, fake) == w4.W4A16_ERR_INVALID_ARG          # Is % 32
    assert block(64, fake, group=128, H=128, I=128) == w4.W4A16_ERR_INVALID_ARG  # Is % group
    assert block(64, fake, group=16) == w4.W4A16_ERR_UNSUPPORTED
    assert block(64, fake, ws=100) == w4.W4A16_ERR_INVALID_ARG  # workspace too small


def test_binding_rejects_host_tensors(w4):
    """Every step runs in the CUDA kernels: host tensors are refused before
    any library call, never computed on the CPU."""
    torch = pytest.importorskip("torch")
    x = torch.zeros((1, 64), dtype=torch.float32)
    qw = torch.zeros((8, 8), dtype=torch.int32)
    sc = torch.zeros((8, 2), dtype=torch.float32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        w4.w4a16_gemm(x, qw, sc)
    with pytest.raises(ValueError, match="CUDA tensor"):
        w4.w4a16_quantize(torch.zeros((8, 64), dtype=torch.float32))
    with pytest.raises(TypeError):
        w4.w4a16_gemm(x.double(), qw, sc)  # neither fp32 nor bf16
    # the MoE layer wrappers check every tensor, the weights and y included
    xm = torch.zeros((2, 64), dtype=torch.float32)
    ids = torch.zeros((2, 1), dtype=torch.int32)
    rw = torch.ones((2, 1), dtype=torch.float32)
    qgu = torch.zeros((1, 64, 8), dtype=torch.int32)
    sgu = torch.zeros((1, 64, 2), dtype=torch.float32)
    qdn = torch.zeros((1, 64, 4), dtype=torch.int32)
    sdn = torch.zeros((1, 64, 1), dtype=torch.float32)
    for fn in (w4.w4a16_moe_gemm, w4.w4a16_moe_gemm_noalloc):
        with pytest.raises(ValueError, match="CUDA tensor"):
            fn(xm, ids, rw, qgu, sgu, qdn, sdn)


def test_package_without_library_fails_to_import(tmp_path):
    """A copy of the package without libw4a16.so raises on import (no fallback)."""
    import shutil
    import subprocess
    import sys
    pkg = os.path.join(ROOT, "int4_w4a16_group_gemm_gb300")
    dst = tmp_path / "int4_w4a16_group_gemm_gb300"
    dst.mkdir()
    shutil.copy(os.path.join(pkg, "__init__.py"), dst / "__init__.py")
    r = subprocess.run([sys.executable, "-c", "import int4_w4a16_group_gemm_gb300"],
                       cwd=tmp_path, capture_output=True, text=True)
    assert r.returncode != 0
    assert "ImportError" in r.stderr and "libw4a16.so" in r.stderr
