"""GPU: the per-(row, 32-column) scale variant -- make_twin_rows and dequant_rows bit-exact
against the oracle, gemm_rows within the GEMM tolerance (bit-exact on one-hot x), the
fused call equal to its repeat, and block exponents repeated over rows giving the block
GEMM's bits."""
import numpy as np
import pytest
import torch

import block_scaled_fp8_weight_gb300 as bsf8
import oracle
from block_scaled_fp8_weight_gb300 import workloads as wl
from _helpers import assert_gemm_close, bf16_bits, same_bits, to_dev_bf16, to_dev_u8

pytestmark = pytest.mark.gpu


def _rows_exact_weight(seed, G=1, N=256, K=1024):
    r = wl.rng(seed)
    w8 = wl.codes(r, (G, N, K))
    w8[..., ::32] = np.where(r.integers(0, 2, size=w8[..., ::32].shape) == 1, 0xFE, 0x7E).astype(np.uint8)
    ex = wl.exponents(r, (G, N, K // 32), 110, 130)
    return w8, ex, oracle.dequant_rows(w8, ex)


def test_make_twin_rows_bit_exact(bsf8_lib):
    """On an exact per-row weight (accepted, the generating twin recovered), on the same
    weight with nudged elements (exactly those segments rejected), and on N(0,1) weights
    (not exact): codes, exponents and flags equal the oracle's bit for bit."""
    w8, ex, w = _rows_exact_weight(71, G=2)
    G, N, K = w.shape
    nudged = wl.apply_nudge(w, [3 * K + 40, N * K + 7 * K + 100])
    normal = wl.activations(wl.rng(72), N, K).reshape(1, N, K)
    for wt in (w, nudged, normal):
        acc, t8, tex, ok = bsf8.make_twin_rows(to_dev_bf16(wt))
        racc, r8, rex, rok = oracle.make_twin_rows(wt)
        assert acc == racc
        assert np.array_equal(t8.cpu().numpy(), r8) and np.array_equal(tex.cpu().numpy(), rex)
        assert np.array_equal(ok.cpu().numpy(), rok)
    acc, t8, tex, _ = bsf8.make_twin_rows(to_dev_bf16(w))
    assert acc and np.array_equal(t8.cpu().numpy(), w8) and np.array_equal(tex.cpu().numpy(), ex)


def test_dequant_rows_all_codes_and_exponents(bsf8_lib):
    """Every code under every exponent byte, one exponent per row: bit-exact."""
    N, K = 256, 256
    w8 = (np.arange(N * K) % 256).astype(np.uint8).reshape(1, N, K)
    ex = (np.arange(N * (K // 32)) % 256).astype(np.uint8).reshape(1, N, K // 32)
    y = bf16_bits(bsf8.dequant_rows(to_dev_u8(w8), to_dev_u8(ex)))
    assert np.all(same_bits(y, oracle.dequant_rows(w8, ex)))


@pytest.mark.parametrize("M,S", [(1, 0), (6, 1), (16, 4), (40, 2)])
def test_gemm_rows_matches_oracle(bsf8_lib, M, S):
    """The draft main_proj-like shape (N = 1280 output rows, K = 5120): sampled rows within
    the GEMM tolerance; repeated calls give the same bits."""
    r = wl.rng(73)
    G, N, K = 1, 1280, 5120
    w8 = wl.codes(r, (G, N, K))
    ex = wl.exponents(r, (G, N, K // 32), 110, 130)
    x = wl.activations(r, M, G * K)
    w8_d, ex_d, x_d = to_dev_u8(w8), to_dev_u8(ex), to_dev_bf16(x)
    y = bf16_bits(bsf8.gemm_rows(x_d, w8_d, ex_d, split_k=S))
    y2 = bf16_bits(bsf8.gemm_rows(x_d, w8_d, ex_d, split_k=S))
    assert bsf8.device_status() == 0
    assert np.array_equal(y, y2)
    assert_gemm_close(y, oracle.gemm_rows(x, w8, ex), f"rows M={M} S={S}")


def test_gemm_rows_one_hot_and_repeated_block_exponents(bsf8_lib):
    """One-hot x over all codes x exponents (one exponent per row): bit-exact.  And with a
    block twin's exponents repeated over rows the per-row GEMM gives the block GEMM's bits
    on the same kernel (the decode-ahead kernel at 6 rows)."""
    M, N, K = 8, 256 * 32, 32
    w8 = (np.arange(N * K) % 256).astype(np.uint8).reshape(1, N, K)
    ex = (np.arange(N) % 256).astype(np.uint8).reshape(1, N, 1)
    for k0 in range(0, K, M):
        x = np.zeros((M, K), dtype=np.uint16)
        x[np.arange(M), (k0 + np.arange(M)) % K] = 0x3F80
        y = bf16_bits(bsf8.gemm_rows(to_dev_bf16(x), to_dev_u8(w8), to_dev_u8(ex), split_k=1))
        assert np.all(same_bits(y, oracle.gemm_rows(x, w8, ex), zero_sign=True))
    wk = wl.WO_A
    bw8, bex = wk.weights()
    x = wk.x(M=6)
    x_d, w8_d = to_dev_bf16(x), to_dev_u8(bw8)
    bsf8.set_option(bsf8.OPT_GEMM_PATH, 4)  # the block GEMM on the decode-ahead kernel too
    try:
        assert bsf8.gemm_kernel(6, wk.N, wk.K, wk.G, 8) == 4
        yb = bf16_bits(bsf8.gemm(x_d, w8_d, to_dev_u8(bex), split_k=8))
    finally:
        bsf8.set_option(bsf8.OPT_GEMM_PATH, 0)
    yr = bf16_bits(bsf8.gemm_rows(x_d, w8_d, to_dev_u8(np.repeat(bex, 32, axis=1)), split_k=8))
    assert np.array_equal(yb, yr)
