"""GPU: bsf8_prefetch_l2 ("docs/tp4-adapters.md", adapter table, l2_prefetch row) is a hint:
the GEMM gives the same bits with or without it, whether the prefetch runs on the GEMM's
stream or on a side stream alongside other work, and the result still matches the oracle."""
import numpy as np
import pytest
import torch

import block_scaled_fp8_weight_gb300 as bsf8
import oracle
from block_scaled_fp8_weight_gb300 import workloads as wl
from _helpers import assert_gemm_close, bf16_bits, to_dev_bf16, to_dev_u8

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("wk,M,S", [(wl.WO_A, 6, 8), (wl.DOWN_PROJ, 6, 0), (wl.TINY, 4, 1)])
def test_prefetch_changes_no_bits(bsf8_lib, wk, M, S):
    w8, ex = wk.weights()
    x = wk.x(M=M)
    w8_d, ex_d, x_d = to_dev_u8(w8), to_dev_u8(ex), to_dev_bf16(x)
    plain = bf16_bits(bsf8.gemm(x_d, w8_d, ex_d, split_k=S))
    bsf8.prefetch_l2(w8_d, ex_d)                        # same stream, right before
    same_stream = bf16_bits(bsf8.gemm(x_d, w8_d, ex_d, split_k=S))
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    bsf8.prefetch_l2(w8_d, ex_d, stream=side)           # side stream, alongside other work
    torch.cuda._sleep(20000)
    overlapped = bf16_bits(bsf8.gemm(x_d, w8_d, ex_d, split_k=S))
    torch.cuda.current_stream().wait_stream(side)
    assert bsf8.device_status() == 0
    assert np.array_equal(plain, same_stream)
    assert np.array_equal(plain, overlapped)
    assert_gemm_close(plain, oracle.gemm(x, w8, ex), wk.name)


def test_prefetch_of_unpadded_exponent_tail(bsf8_lib):
    """Exponent arrays whose size is not a multiple of 16 bytes (5120 x 576: 2880 bytes):
    the prefetch covers the 16-byte-aligned part and the GEMM is unaffected."""
    r = wl.rng(5)
    G, N, K = 1, 96, 160                                 # 3 x 5 = 15 exponent bytes
    w8s = wl.codes(r, (G, N, K))
    exs = wl.exponents(r, (G, N // 32, K // 32), 115, 127)
    x = wl.activations(r, 3, K)
    w8_d, ex_d = to_dev_u8(w8s), to_dev_u8(exs)
    bsf8.prefetch_l2(w8_d, ex_d)
    y = bf16_bits(bsf8.gemm(to_dev_bf16(x), w8_d, ex_d, split_k=1))
    assert bsf8.device_status() == 0
    assert_gemm_close(y, oracle.gemm(x, w8s, exs))
