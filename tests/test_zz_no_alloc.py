"""bsf8_gemm_static_scratch: the GEMM for callers that cannot allocate device memory.

Callers such as a serving engine that has reserved all GPU memory for its own arena (or a
plugin running inside one) have no workspace to give.  Where bsf8_gemm needs no workspace
this entry point is bsf8_gemm; otherwise it keeps the split-K partials in a buffer compiled
into the library.  The tests call it through the C ABI, several calls in a row on
different inputs, on both routes (calls whose kernels sum the splits on chip, and calls that
write partials), and check each result against the CPU oracle within the GEMM tolerance of
the other tests, and bit for bit against bsf8_gemm (which runs the same kernel and sums the
splits in the same order); the automatic split (split_k = 0) is covered, and so are partials
of exactly the buffer's size and just past it.  The file is named so that pytest collects it
last.
"""
import ctypes

import numpy as np
import pytest
import torch

import block_scaled_fp8_weight_gb300 as bsf8
import oracle
from block_scaled_fp8_weight_gb300 import workloads as wl
from _helpers import assert_gemm_close, bf16_bits, to_dev_bf16, to_dev_u8

pytestmark = pytest.mark.gpu

STATIC_SCRATCH_BYTES = 8 * 1024 * 1024
OK, ERR_WORKSPACE = 0, 4


def _entry(lib):
    fn = lib.bsf8_gemm_static_scratch
    P, I, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    fn.argtypes = [P, P, P, P, I, I, I, I, I, I64, P]
    fn.restype = I
    return fn


def _call(fn, x_d, w8_d, ex_d, y_d, M, N, K, G, S):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return fn(ctypes.c_void_p(x_d.data_ptr()), ctypes.c_void_p(w8_d.data_ptr()),
              ctypes.c_void_p(ex_d.data_ptr()), ctypes.c_void_p(y_d.data_ptr()),
              M, N, K, G, S, x_d.stride(0), stream)


def test_static_scratch_gemm_matches_oracle_and_bsf8_gemm(bsf8_lib):
    fn = _entry(bsf8_lib)
    # on chip (no workspace): wo_a, down_proj and tiny decode calls, the mid-row weight at
    # 192 tokens in 4 splits (summed in a cluster); with partials in the buffer: gate_up and
    # the mid-row weight in 16 splits
    cases = [(wl.WO_A, 6, 8, False), (wl.DOWN_PROJ, 6, 4, False), (wl.WO_A, 6, 0, False),
             (wl.DOWN_PROJ, 6, 0, False), (wl.TINY, 4, 4, False), (wl.MID, 192, 4, False),
             (wl.GATE_UP, 64, 16, True), (wl.MID, 32, 16, True)]
    for wk, M, S, partials in cases:             # calls in a row, different inputs
        assert (bsf8.workspace_bytes(M, wk.N, wk.K, wk.G, S) > 0) == partials, (wk.name, M, S)
        w8, ex = wk.weights()
        x = wk.x(M=M)
        w8_d, ex_d, x_d = to_dev_u8(w8), to_dev_u8(ex), to_dev_bf16(x)
        S_used = S or bsf8.auto_split(M, wk.N, wk.K, wk.G)
        if partials:
            assert S_used * M * wk.G * wk.N * 4 <= STATIC_SCRATCH_BYTES
        y_d = torch.empty((M, wk.G, wk.N), dtype=torch.bfloat16, device="cuda")
        assert _call(fn, x_d, w8_d, ex_d, y_d, M, wk.N, wk.K, wk.G, S) == OK
        ref = bf16_bits(bsf8.gemm(x_d, w8_d, ex_d, split_k=S))
        assert bsf8.device_status() == 0
        got = bf16_bits(y_d)
        assert np.array_equal(got, ref), f"{wk.name} S={S}"
        rows = list(range(M)) if M <= 8 else sorted({0, M // 2, M - 1})
        assert_gemm_close(got[rows], oracle.gemm(x[rows], w8, ex), f"{wk.name} M={M} S={S}")


def test_static_scratch_at_and_past_its_size(bsf8_lib):
    """Partials of exactly 8 MiB run (S = 16, M = 64, G = 1, N = 2048: 16*64*2048*4 bytes;
    more than 8 splits, so bsf8_gemm too writes partials); one more token row is refused
    with BSF8_ERR_WORKSPACE and writes nothing."""
    fn = _entry(bsf8_lib)
    G, N, K, S = 1, 2048, 4096, 16
    r = wl.rng(8 << 20)
    w8 = wl.codes(r, (G, N, K))
    ex = wl.exponents(r, (G, N // 32, K // 32), 115, 127)
    w8_d, ex_d = to_dev_u8(w8), to_dev_u8(ex)
    M = 64
    assert S * M * G * N * 4 == STATIC_SCRATCH_BYTES
    assert bsf8.workspace_bytes(M, N, K, G, S) == STATIC_SCRATCH_BYTES
    x = wl.activations(r, M, G * K)
    x_d = to_dev_bf16(x)
    y_d = torch.empty((M, G, N), dtype=torch.bfloat16, device="cuda")
    assert _call(fn, x_d, w8_d, ex_d, y_d, M, N, K, G, S) == OK
    ref = bf16_bits(bsf8.gemm(x_d, w8_d, ex_d, split_k=S))
    assert bsf8.device_status() == 0
    got = bf16_bits(y_d)
    assert np.array_equal(got, ref)
    rows = [0, 33, M - 1]
    assert_gemm_close(got[rows], oracle.gemm(x[rows], w8, ex), "8 MiB of partials")

    M1 = M + 1
    x1_d = to_dev_bf16(wl.activations(r, M1, G * K))
    y1_d = torch.full((M1, G, N), 3.0, dtype=torch.bfloat16, device="cuda")
    assert _call(fn, x1_d, w8_d, ex_d, y1_d, M1, N, K, G, S) == ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(y1_d == 3.0)


def test_static_scratch_rejects_partials_far_beyond_its_size(bsf8_lib):
    fn = _entry(bsf8_lib)
    wk = wl.MID                                   # G=4, N=1024, K=4096
    M, S = 192, 8                                 # 8*192*4*1024*4 B = 25 MiB > 8 MiB
    w8, ex = wk.weights()
    x_d = to_dev_bf16(wk.x(M=M))
    y_d = torch.empty((M, wk.G, wk.N), dtype=torch.bfloat16, device="cuda")
    assert _call(fn, x_d, to_dev_u8(w8), to_dev_u8(ex), y_d, M, wk.N, wk.K, wk.G, S) == ERR_WORKSPACE
