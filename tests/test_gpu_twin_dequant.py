"""GPU parity of bsf8_dequant and bsf8_make_twin against the CPU oracle: both are
integer/byte results (codes, exponent bytes, flags) or exact bf16 values, so the bar is
bit-exact (any NaN matches any NaN)."""
import numpy as np
import pytest
import torch

import block_scaled_fp8_weight_gb300 as bsf8
import oracle
from block_scaled_fp8_weight_gb300 import workloads as wl
from _helpers import bf16_bits, same_bits, to_dev_bf16, to_dev_u8

pytestmark = pytest.mark.gpu


def exhaustive_twin_rows():
    """W [1, 8192, 32]: row block b has exponent byte b (all 256), and its 1024 codes
    cover every byte value four times."""
    N, K = 256 * 32, 32
    codes = (np.arange(N * K) % 256).astype(np.uint8).reshape(1, N, K)
    ex = np.arange(256, dtype=np.uint8).reshape(1, 256, 1)
    return codes, ex


def exhaustive_twin_cols():
    """W [1, 32, 8192]: block column b has exponent byte b; codes cover all 256."""
    N, K = 32, 256 * 32
    codes = np.zeros((1, N, K), dtype=np.uint8)
    for b in range(256):
        codes[0, :, b * 32:(b + 1) * 32] = (np.arange(1024) % 256).reshape(32, 32)
    ex = np.arange(256, dtype=np.uint8).reshape(1, 1, 256)
    return codes, ex


@pytest.mark.parametrize("layout", [exhaustive_twin_rows, exhaustive_twin_cols])
def test_dequant_every_code_and_exponent(bsf8_lib, layout):
    w8, ex = layout()
    got = bf16_bits(bsf8.dequant(to_dev_u8(w8), to_dev_u8(ex)))
    ref = oracle.dequant(w8, ex)
    assert np.all(same_bits(got, ref))


@pytest.mark.parametrize("wk", [wl.TINY, wl.WO_A, wl.DOWN_PROJ])
def test_dequant_workloads(bsf8_lib, wk):
    w8, ex = wk.weights()
    got = bf16_bits(bsf8.dequant(to_dev_u8(w8), to_dev_u8(ex)))
    assert np.array_equal(got, oracle.dequant(w8, ex))


def _twin_compare(w_bits):
    acc_o, w8_o, ex_o, ok_o = oracle.make_twin(w_bits)
    acc_g, w8_g, ex_g, ok_g = bsf8.make_twin(to_dev_bf16(w_bits))
    w8_g, ex_g, ok_g = w8_g.cpu().numpy(), ex_g.cpu().numpy(), ok_g.cpu().numpy()
    assert np.array_equal(ex_g, ex_o)
    assert np.array_equal(ok_g, ok_o)
    assert np.array_equal(w8_g, w8_o), np.argwhere(w8_g != w8_o)[:5]
    assert acc_g == acc_o
    return acc_g


def test_make_twin_exact_weights_accept_and_round_trip(bsf8_lib):
    w8, ex = wl.TINY.weights()
    w = oracle.dequant(w8, ex)
    assert _twin_compare(w)
    tw = bsf8.twin_or_none(to_dev_bf16(w))
    back = bf16_bits(bsf8.dequant(*tw))
    assert np.all(same_bits(back, w, zero_sign=True))


def test_make_twin_nudged_weights_rejected(bsf8_lib):
    w8, ex = wl.TINY.weights()
    w = oracle.dequant(w8, ex)
    G, N, K = w.shape
    wn = wl.apply_nudge(w, wl.nudge_sites(wl.rng(5), G, N, K))
    assert not _twin_compare(wn)
    assert bsf8.twin_or_none(to_dev_bf16(wn)) is None


def test_make_twin_wo_a_shape(bsf8_lib):
    w8, ex = wl.WO_A.weights()
    w = oracle.dequant(w8, ex)
    assert _twin_compare(w)


def test_make_twin_random_non_exact_weights(bsf8_lib):
    """N(0,1) weights exercise the nearest-even e4m3 rounding on arbitrary values."""
    r = wl.rng(21)
    w = wl.activations(r, 3 * 128, 256).reshape(3, 128, 256)
    assert not _twin_compare(w)


def test_make_twin_special_blocks(bsf8_lib):
    r = wl.rng(22)
    w = wl.activations(r, 64, 32 * 12).reshape(1, 64, 32 * 12)
    blk = lambda j: (slice(0, 32), slice(32 * j, 32 * j + 32))
    w[0][blk(0)] = 0x0000                                  # all +0
    w[0][blk(1)] = 0x8000                                  # all -0
    w[0][blk(2)] = w[0][blk(2)] & 0x807F                   # bf16 subnormals only
    w[0][blk(3)] = w[0][blk(3)] | 0x7F00                   # huge values (some inf/nan)
    w[0][blk(4)] = (w[0][blk(4)] & 0x80FF) | 0x7E00        # huge finite
    w[0][5, 32 * 5 + 3] = 0x7F80                           # one +inf
    w[0][7, 32 * 6 + 9] = 0xFFC1                           # one NaN
    w[0][blk(7)] = (w[0][blk(7)] & 0x807F) | 0x0080       # around 2^-126
    w[0][blk(8)] = 0x43E0                                  # all 448
    w[0][blk(9)] = 0x43E1                                  # all 450
    w[0][blk(10)] = (w[0][blk(10)] & 0x8000) | 0x0001      # +-min subnormal
    _twin_compare(w)


def test_make_twin_all_bf16_patterns(bsf8_lib):
    """Every finite bf16 pattern as an element, with block maxima spread over the range."""
    pats = np.arange(0x10000, dtype=np.uint32).astype(np.uint16)
    pats = pats[(pats & 0x7FFF) < 0x7F80]
    n = (pats.size + 1023) // 1024 * 1024
    w = np.zeros(n, dtype=np.uint16)
    w[:pats.size] = wl.rng(23).permutation(pats)
    _twin_compare(w.reshape(1, n // 32, 32))
