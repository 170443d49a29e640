"""GPU: the wide-weight kernel (BSF8_OPT_GEMM_PATH 6, up to 8 token rows) against the
CPU oracle -- on its f16 path, on its bf16-rebuild path and where both meet in one row.

The kernel takes the f16 path for a 32 x 32 block when the exponent byte is in
[16, 200] and every token row's activations convert to f16 exactly after the row's
power-of-two scale; other blocks take the exact bf16 rebuild.  Outputs are held to the
GEMM's floating-point bar per token row and exponent band (max |y - y_ref| <= 1e-2 *
rms(y_ref), >= 99.9% within 1 bf16 ulp), non-finite outputs must match the oracle's
class exactly (NaN, +inf, -inf), and results are bitwise reproducible."""
import numpy as np
import pytest
import torch

import block_scaled_fp8_weight_gb300 as bsf8
import oracle
from block_scaled_fp8_weight_gb300 import workloads as wl
from _helpers import assert_gemm_close, bf16_bits, is_nan_bits, same_bits, to_dev_bf16, to_dev_u8

pytestmark = pytest.mark.gpu

WIDE = 6


def bf16_of(f):
    return torch.from_numpy(np.asarray(f, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def run_wide(x, w8, ex, S):
    w8_d, ex_d, x_d = to_dev_u8(w8), to_dev_u8(ex), to_dev_bf16(x)
    bsf8.set_option(bsf8.OPT_GEMM_PATH, WIDE)
    try:
        y = bf16_bits(bsf8.gemm(x_d, w8_d, ex_d, split_k=S))
        y2 = bf16_bits(bsf8.gemm(x_d, w8_d, ex_d, split_k=S))
        two = bf16_bits(bsf8.splitk_reduce(bsf8.gemm_partials(x_d, w8_d, ex_d, S)))
        assert bsf8.device_status() == 0
    finally:
        bsf8.set_option(bsf8.OPT_GEMM_PATH, 0)
    assert np.array_equal(y, y2)
    assert np.array_equal(y, two)
    return y


def assert_rows_close(y, ref, row_groups, what):
    """Per token row and weight-row group: non-finite classes equal, finite ones within
    the tolerance of that row's own scale."""
    y = np.asarray(y)
    ref = np.asarray(ref)
    fin = (ref & 0x7F80) != 0x7F80
    # NaN where the oracle has NaN, the same infinity where it has one
    assert np.array_equal(is_nan_bits(y), is_nan_bits(ref)), f"{what}: NaN pattern"
    inf = ~fin & ~is_nan_bits(ref)
    assert np.array_equal(y[inf], ref[inf]), f"{what}: infinities"
    M = y.shape[0]
    for m in range(M):
        for g0, g1 in row_groups:
            ys, rs = y[m, :, g0:g1], ref[m, :, g0:g1]
            ok = ((rs & 0x7F80) != 0x7F80)
            if ok.sum() == 0:
                continue
            assert_gemm_close(ys[ok], rs[ok], f"{what} m={m} rows {g0}:{g1}")


def test_one_hot_every_code_and_exponent(bsf8_lib):
    """x rows are unit vectors, so every output is one exact product: the wide-weight
    kernel must reproduce the oracle bit for bit (zeros by value, NaN as NaN) for all 256
    codes x 256 exponent bytes -- bytes 16..200 on the f16 path, the rest on the rebuild."""
    M, N, K = 8, 256 * 32, 128
    w8 = (np.arange(N * K) % 256).astype(np.uint8).reshape(1, N, K)
    ex = np.repeat(np.arange(256, dtype=np.uint8).reshape(1, 256, 1), K // 32, axis=2)
    w8_d, ex_d = to_dev_u8(w8), to_dev_u8(ex)
    bsf8.set_option(bsf8.OPT_GEMM_PATH, WIDE)
    try:
        for k0 in range(0, K, M):
            x = np.zeros((M, K), dtype=np.uint16)
            for m in range(M):
                x[m, (k0 + m) % K] = 0x3F80
            y = bf16_bits(bsf8.gemm(to_dev_bf16(x), w8_d, ex_d, split_k=1))
            assert np.all(same_bits(y, oracle.gemm(x, w8, ex), zero_sign=True)), k0
    finally:
        bsf8.set_option(bsf8.OPT_GEMM_PATH, 0)


@pytest.mark.parametrize("M,S", [(1, 1), (5, 1), (8, 3), (6, 4)])
def test_exponent_bands_mix_both_paths(bsf8_lib, M, S):
    """Row blocks whose exponent bytes straddle the f16 window at both ends ([8, 24] and
    [192, 208]) next to ones inside it: within a row, blocks alternate between the two
    paths, and every row band matches the oracle at its own scale."""
    r = wl.rng(301)
    G, N, K = 2, 384, 1536
    w8 = wl.codes(r, (G, N, K))
    ex = np.empty((G, N // 32, K // 32), dtype=np.uint8)
    bands = [(8, 24), (115, 127), (192, 208)]
    for nb in range(N // 32):
        lo, hi = bands[nb % 3]
        ex[:, nb, :] = wl.exponents(r, (G, K // 32), lo, hi)
    x = wl.activations(r, M, G * K)
    y = run_wide(x, w8, ex, S)
    ref = oracle.gemm(x, w8, ex)
    groups = [(32 * nb, 32 * nb + 32) for nb in range(N // 32)]
    assert_rows_close(y, ref, groups, f"bands M={M} S={S}")


def test_activation_scales_on_the_f16_path(bsf8_lib):
    """Token rows whose scales sit near the ends of the f16 path's range (largest |x|
    near 2^102 and 2^-78), a row with activations 2^-40 below its largest in some blocks
    (those blocks fall back to the rebuild), an all-zero row and ordinary rows."""
    r = wl.rng(302)
    G, N, K = 1, 256, 2048
    w8 = wl.codes(r, (G, N, K))
    ex = wl.exponents(r, (G, N // 32, K // 32), 115, 127)
    xf = r.standard_normal(size=(6, K)).astype(np.float32)
    xf[1] *= 2.0 ** 100
    xf[2] *= 2.0 ** -80
    xf[3, ::97] *= 2.0 ** -40
    xf[4] = 0.0
    x = bf16_of(xf)
    y = run_wide(x, w8, ex, 1)
    ref = oracle.gemm(x, w8, ex)
    assert_rows_close(y, ref, [(0, N)], "f16 scales")
    assert np.all(y[4] == 0)  # zero activations: +0 (sums start at +0)


def test_activation_rows_outside_the_f16_path(bsf8_lib):
    """Rows that send every block to the rebuild: largest |x| near 2^122 and 2^-93 (scale
    outside [-100, 100]), a row holding +inf, one holding NaN -- with an ordinary row that
    shares their MMAs.  Exponent bytes 100..110 keep every product finite (with larger
    weights the 2^120 row overflows single products, and whether a sum of overflowed
    products is an infinity or NaN then depends on the order of the sum)."""
    r = wl.rng(304)
    G, N, K = 1, 256, 2048
    w8 = wl.codes(r, (G, N, K))
    ex = wl.exponents(r, (G, N // 32, K // 32), 100, 110)
    xf = r.standard_normal(size=(5, K)).astype(np.float32)
    xf[1] *= 2.0 ** 120
    xf[2] *= 2.0 ** -95
    xf[3, 700] = np.inf
    xf[4, 1500] = np.nan
    x = bf16_of(xf)
    y = run_wide(x, w8, ex, 1)
    ref = oracle.gemm(x, w8, ex)
    assert_rows_close(y, ref, [(0, N)], "rebuild rows")


def test_nan_codes_poison_their_rows_on_both_paths(bsf8_lib):
    """e4m3 NaN codes (0x7F / 0xFF) in blocks on the f16 path (exponent 120) and on the
    rebuild path (exponent 3): exactly the rows holding one are NaN, for every token."""
    r = wl.rng(303)
    G, N, K = 1, 256, 1024
    w8 = wl.codes(r, (G, N, K))
    ex = wl.exponents(r, (G, N // 32, K // 32), 118, 122)
    ex[0, 1::2, 5] = 3
    sites = [(7, 5 * 32 + 3), (40, 5 * 32 + 30), (100, 900), (255, 0)]
    for n, k in sites:
        w8[0, n, k] = 0x7F if (n % 2) else 0xFF
    x = wl.activations(r, 6, K)
    y = run_wide(x, w8, ex, 2)
    ref = oracle.gemm(x, w8, ex)
    assert np.array_equal(is_nan_bits(y), is_nan_bits(ref))
    assert is_nan_bits(y[:, 0, 7]).all() and is_nan_bits(y[:, 0, 255]).all()
    keep = np.ones(N, dtype=bool)
    keep[[n for n, _ in sites]] = False
    assert_gemm_close(y[:, :, keep], ref[:, :, keep], "nan codes")


@pytest.mark.parametrize("M", [1, 6, 8])
def test_head_full_size_sampled(bsf8_lib, M):
    """The head-like weight (N = 32768, K = 5120, 128-row tasks over all SMs) through the
    wide-weight kernel: the last 2048 rows against the oracle."""
    wk = wl.HEAD
    w8, ex = wk.weights()
    x = wk.x(M=M)
    y = run_wide(x, w8, ex, 1)
    n0 = wk.N - 2048
    ref = oracle.gemm(x, w8[:, n0:], ex[:, n0 // 32:])
    assert_gemm_close(y[:, :, n0:], ref, f"head M={M}")
