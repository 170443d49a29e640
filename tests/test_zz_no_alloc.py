"""bsf8_gemm_static_scratch: the GEMM for callers that cannot allocate device memory.

Callers such as a serving engine that has reserved all GPU memory for its own arena (or a
plugin running inside one) have no workspace to give; this entry point keeps its split-K
partials in a buffer compiled into the library instead.  The test calls it through the C
ABI, twice in a row on different inputs, and checks each result against bsf8_gemm within
the GEMM tolerance of the other tests.  The file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import block_scaled_fp8_weight_gb300 as bsf8
from block_scaled_fp8_weight_gb300 import workloads as wl
from _helpers import assert_gemm_close, bf16_bits, to_dev_bf16, to_dev_u8

pytestmark = pytest.mark.gpu

STATIC_SCRATCH_BYTES = 8 * 1024 * 1024
ERR_WORKSPACE = 4


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


def test_static_scratch_gemm_matches_bsf8_gemm_on_two_calls(bsf8_lib):
    fn = _entry(bsf8_lib)
    cases = [(wl.WO_A, 6, 8), (wl.DOWN_PROJ, 6, 4)]
    for wk, M, S in cases:                       # two calls in a row, different inputs
        w8, ex = wk.weights()
        x = wk.x(M=M)
        w8_d, ex_d, x_d = to_dev_u8(w8), to_dev_u8(ex), to_dev_bf16(x)
        assert S * M * wk.G * wk.N * 4 <= STATIC_SCRATCH_BYTES
        y_d = torch.empty((M, wk.G, wk.N), dtype=torch.bfloat16, device="cuda")
        assert _call(fn, x_d, w8_d, ex_d, y_d, M, wk.N, wk.K, wk.G, S) == 0
        ref = bf16_bits(bsf8.gemm(x_d, w8_d, ex_d, split_k=S))
        assert bsf8.device_status() == 0
        assert_gemm_close(bf16_bits(y_d), ref, f"{wk.name} S={S}")


def test_static_scratch_rejects_partials_beyond_its_size(bsf8_lib):
    fn = _entry(bsf8_lib)
    wk = wl.MID                                   # G=4, N=1024, K=4096
    M, S = 192, 8                                 # 8*192*4*1024*4 B = 25 MiB > 8 MiB
    w8, ex = wk.weights()
    x_d = to_dev_bf16(wk.x(M=M))
    y_d = torch.empty((M, wk.G, wk.N), dtype=torch.bfloat16, device="cuda")
    assert _call(fn, x_d, to_dev_u8(w8), to_dev_u8(ex), y_d, M, wk.N, wk.K, wk.G, S) == ERR_WORKSPACE
