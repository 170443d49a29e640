"""Host-side checks of the C ABI: no GPU needed, no kernel launched.

* libbsf8.so loads and exports every function include/bsf8.h declares;
* every entry point rejects invalid arguments with the documented status code before
  any CUDA call (fake device addresses are only ever paired with an invalid argument,
  so nothing can reach a kernel even where a GPU is present);
* the pure-host helpers (workspace size, automatic split count, options, strerror).
"""
import ctypes
import os
import re

import pytest

import block_scaled_fp8_weight_gb300 as bsf8
from block_scaled_fp8_weight_gb300 import build as bsf8_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bsf8.h")

OK, SHAPE, ALIGN, STRIDE, WORKSPACE, NULL, CUDA, TIMEOUT, DEVICE, VALUE = range(10)

A = 0x10000        # a 16-byte aligned fake device address (never dereferenced here)
B = 0x20000
C = 0x30000
D = 0x40000


@pytest.fixture(scope="module")
def lib():
    bsf8_build.build()
    return bsf8.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bsf8_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_path_entry_points():
    names = declared_functions()
    for need in ("bsf8_make_twin", "bsf8_dequant", "bsf8_gemm", "bsf8_pad_k", "bsf8_pad_x",
                 "bsf8_gemm_partials", "bsf8_splitk_reduce", "bsf8_gemm_workspace_bytes"):
        assert need in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(bsf8_build.LIB)
    missing = [n for n in declared_functions() if not hasattr(raw, n)]
    assert not missing, missing


def test_strerror_and_version(lib):
    for code in range(10):
        assert lib.bsf8_strerror(code)
    assert lib.bsf8_strerror(99) == b"unknown status"
    assert lib.bsf8_version() >= 100


def _gemm(lib, x=A, w8=B, ex=C, y=D, M=6, N=1024, K=4096, G=2, S=8, ldx=None, ws=0, wsb=0):
    ldx = G * K if ldx is None else ldx
    return lib.bsf8_gemm(x, w8, ex, y, M, N, K, G, S, ldx, ws, wsb, None)


def test_gemm_validation(lib):
    assert _gemm(lib, x=0) == NULL
    assert _gemm(lib, y=0) == NULL
    assert _gemm(lib, M=0) == SHAPE
    assert _gemm(lib, M=16385) == SHAPE  # past BSF8_MAX_M
    assert _gemm(lib, N=1000) == SHAPE
    assert _gemm(lib, K=4016) == SHAPE          # 4016 = 125.5 * 32
    assert _gemm(lib, G=0) == SHAPE
    assert _gemm(lib, S=-1) == SHAPE
    assert _gemm(lib, S=129) == SHAPE          # > K/32
    assert _gemm(lib, ldx=2 * 4096 - 8) == STRIDE
    assert _gemm(lib, x=A + 2) == ALIGN
    assert _gemm(lib, w8=B + 8) == ALIGN
    assert _gemm(lib, ldx=2 * 4096 + 4) == ALIGN
    # more than 64 column tasks per 16-row slab run through the workspace: a missing or
    # short workspace is rejected
    assert _gemm(lib, S=128) == WORKSPACE
    need = lib.bsf8_gemm_workspace_bytes(6, 1024, 4096, 2, 128)
    assert need == 128 * 6 * 2 * 1024 * 4
    assert _gemm(lib, S=128, ws=A, wsb=need - 1) == WORKSPACE
    assert _gemm(lib, S=128, ws=A + 4, wsb=need) == ALIGN


def test_partials_reduce_pad_validation(lib):
    gp = lib.bsf8_gemm_partials
    assert gp(A, B, C, 0, 6, 1024, 4096, 2, 8, 8192, None) == NULL
    assert gp(A, B, C, D, 6, 1024, 4096, 2, 0, 8192, None) == SHAPE   # explicit S >= 1
    assert gp(A, B, C, D + 4, 6, 1024, 4096, 2, 8, 8192, None) == ALIGN
    assert lib.bsf8_splitk_reduce(A, B, 0, 10, None) == SHAPE
    assert lib.bsf8_splitk_reduce(A, B, 2, -1, None) == SHAPE
    assert lib.bsf8_splitk_reduce(0, B, 2, 10, None) == NULL
    assert lib.bsf8_splitk_reduce(0, 0, 2, 0, None) == OK                # nothing to do
    pk = lib.bsf8_pad_k
    assert pk(A, B, C, 0, 1, 5120, 576, 640, 127, None) == NULL
    assert pk(A, B, C, D, 1, 5120, 576, 620, 127, None) == SHAPE
    assert pk(A, B, C, D, 1, 5120, 576, 544, 127, None) == SHAPE
    assert pk(A, B, C, D, 1, 5120, 576, 640, 256, None) == VALUE
    assert pk(A, B, C, D, 1, 5120, 576, 640, -1, None) == VALUE
    assert pk(A + 1, B, C, D, 1, 5120, 576, 640, 127, None) == ALIGN
    px = lib.bsf8_pad_x
    assert px(0, 576, B, 6, 1, 576, 640, None) == NULL
    assert px(A, 560, B, 6, 1, 576, 640, None) == STRIDE
    assert px(A, 580, B, 6, 1, 576, 640, None) == ALIGN
    assert px(A, 576, B, 6, 1, 576, 600, None) == SHAPE
    assert px(A, 576, B, 0, 1, 576, 640, None) == SHAPE


def test_twin_and_dequant_validation(lib):
    mt = lib.bsf8_make_twin
    assert mt(0, B, C, 0, D, 1, 256, 512, None) == NULL
    assert mt(A, B, C, 0, 0, 1, 256, 512, None) == NULL
    assert mt(A, B, C, 0, D, 1, 250, 512, None) == SHAPE
    assert mt(A + 2, B, C, 0, D, 1, 256, 512, None) == ALIGN
    dq = lib.bsf8_dequant
    assert dq(A, B, 0, 1, 256, 512, None) == NULL
    assert dq(A, B, C, 1, 256, 500, None) == SHAPE
    assert dq(A, B, C + 2, 1, 256, 512, None) == ALIGN


def test_workspace_and_auto_split(lib):
    # up to 64 column tasks per slab are summed on chip: no workspace
    for S in (0, 1, 8, 9, 16, 64):
        assert lib.bsf8_gemm_workspace_bytes(6, 1024, 4096, 2, S) == 0, S
    assert lib.bsf8_gemm_workspace_bytes(6, 1024, 4096, 2, 65) == 65 * 6 * 2 * 1024 * 4
    # very long splits need more than 8 tasks each: K = 65536 in 16 splits
    assert lib.bsf8_gemm_workspace_bytes(6, 64, 65536, 1, 16) == 16 * 6 * 64 * 4
    # up to 8 token rows: one split (the kernels cut it into column tasks themselves; for
    # wo_a one split sums its 8 tasks in the same left-to-right order as the page's 8 splits)
    assert lib.bsf8_gemm_auto_split(6, 1024, 4096, 2) == 1
    assert lib.bsf8_gemm_auto_split(6, 32768, 5120, 1) == 1
    # 9..16 rows: one split too (the streaming and decode-ahead tensor-core kernels cut it
    # into column tasks; extra splits measured no faster on the streaming kernel)
    assert lib.bsf8_gemm_auto_split(12, 1024, 4096, 2) == 1
    assert lib.bsf8_gemm_auto_split(16, 1024, 4096, 4) == 1
    # past 16 rows, never more splits than 32-column blocks
    assert lib.bsf8_gemm_auto_split(64, 32, 64, 1) == 2
    assert lib.bsf8_gemm_auto_split(0, 1024, 4096, 2) == -SHAPE
    for M in (1, 2, 8, 9, 64, 192):
        s = lib.bsf8_gemm_auto_split(M, 5120, 576, 1)
        assert 1 <= s <= 8


def test_gemm_kernel_query_validation(lib):
    """bsf8_gemm_kernel: invalid sizes give -BSF8_ERR_SHAPE; a forced kernel that cannot run
    the call gives -BSF8_ERR_VALUE (host logic only); the kernels removed from the library
    (1, 3) and unknown values cannot be forced."""
    q = lib.bsf8_gemm_kernel
    assert q(0, 1024, 4096, 2, 8) == -SHAPE
    assert q(6, 1000, 4096, 2, 8) == -SHAPE
    assert q(6, 1024, 4096, 2, 129) == -SHAPE
    try:
        assert lib.bsf8_set_option(4, 4) == OK           # decode-ahead: up to 8 rows
        assert q(12, 1024, 4096, 2, 8) == -VALUE
        assert q(6, 1024, 4096, 2, 8) == 4
        assert lib.bsf8_set_option(4, 6) == OK           # wide-weight: 128-column splits
        assert q(6, 5120, 576, 1, 1) == -VALUE
        assert lib.bsf8_set_option(4, 2) == OK           # streaming: any call
        assert q(100, 1024, 4096, 2, 3) == 2
        for bad in (1, 3, 8):
            assert lib.bsf8_set_option(4, bad) == VALUE
    finally:
        lib.bsf8_set_option(4, 0)
    # a refused forced kernel is refused by the GEMM entry points too, before any CUDA call
    try:
        assert lib.bsf8_set_option(4, 4) == OK
        assert _gemm(lib, M=12) == VALUE
        assert lib.bsf8_gemm_partials(A, B, C, D, 12, 1024, 4096, 2, 8, 8192, None) == VALUE
    finally:
        lib.bsf8_set_option(4, 0)


def test_prefetch_l2_validation(lib):
    pf = lib.bsf8_prefetch_l2
    assert pf(0, B, 2, 1024, 4096, None) == NULL
    assert pf(A, 0, 2, 1024, 4096, None) == NULL
    assert pf(A, B, 2, 1000, 4096, None) == SHAPE
    assert pf(A, B, 0, 1024, 4096, None) == SHAPE
    assert pf(A + 8, B, 2, 1024, 4096, None) == ALIGN
    assert pf(A, B + 1, 2, 1024, 4096, None) == ALIGN


def test_sm_clock_sample_validation(lib):
    """The measurement aid rejects a NULL buffer and SM counts out of range before any launch."""
    assert lib.bsf8_sm_clock_sample(0, 152, None) == NULL
    assert lib.bsf8_sm_clock_sample(A, 0, None) == SHAPE
    assert lib.bsf8_sm_clock_sample(A, 4097, None) == SHAPE


def test_options_roundtrip(lib):
    assert lib.bsf8_get_option(1) == 1
    assert lib.bsf8_set_option(1, 0) == OK and lib.bsf8_get_option(1) == 0
    assert lib.bsf8_set_option(1, 1) == OK
    old = lib.bsf8_get_option(2)
    assert lib.bsf8_set_option(2, 12345) == OK and lib.bsf8_get_option(2) == 12345
    assert lib.bsf8_set_option(2, old) == OK
    assert lib.bsf8_set_option(42, 1) == VALUE
    assert lib.bsf8_set_option(2, -5) == VALUE
    assert lib.bsf8_get_option(42) == -VALUE


def test_binding_rejects_cpu_tensors():
    torch = pytest.importorskip("torch")
    w8 = torch.zeros((1, 32, 32), dtype=torch.uint8)
    ex = torch.zeros((1, 1, 1), dtype=torch.uint8)
    with pytest.raises(ValueError, match="CUDA tensor"):
        bsf8.dequant(w8, ex)

