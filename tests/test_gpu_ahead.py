"""GPU: the decode-ahead tensor-core kernel (BSF8_OPT_GEMM_PATH 7, up to 32 token rows)
against the CPU oracle.

A block holds 128 weight rows x at most 512 columns of one split, the first 128 columns'
weights in shared memory and the rest in tensor memory as the MMA's A operand; a cluster
holds all tasks of its rows (S splits x tps tasks <= 8) and folds them in split order.
The cases cover both A sources, clusters of 1 to 16 blocks (3, 5, 7, 10, 12, 14 included), weight
rows past N inside a 128-row block, an empty split, every code under every exponent byte,
NaN codes, per-row exponents and the head-to-toe wo_a shape.  Outputs are held to the
GEMM's floating-point bar; repeated calls and gemm = reduce(partials) are bitwise equal."""
import numpy as np
import pytest

import block_scaled_fp8_weight_gb300 as bsf8
import oracle
from block_scaled_fp8_weight_gb300 import workloads as wl
from _helpers import assert_gemm_close, bf16_bits, is_nan_bits, same_bits, to_dev_bf16, to_dev_u8

pytestmark = pytest.mark.gpu

AHEAD = 7


def plan_holds(M, K, S):
    """The kernel's plan rule (bsf8_ahead.cu, plan_ahead): tasks of at most 512 columns,
    S x tasks-per-split blocks in a cluster of at most 16 (past 8 where the GPU schedules
    such clusters, as a GB300 does), at most 32 token rows.  Cases
    that fail it would silently run on another kernel, so every case asserts it."""
    chunk = -(-(K // 32) // S) * 32
    tps = max(1, -(-chunk // 512))
    kt = -(-(-(-chunk // tps)) // 32) * 32
    ntok = 16 if M <= 16 else 32
    return 1 <= M <= 32 and S * tps <= 16 and kt <= 512 and 64 + max(0, kt - 128) // 2 <= 256


def run_ahead(x, w8, ex, S, rows=False):
    w8_d, ex_d, x_d = to_dev_u8(w8), to_dev_u8(ex), to_dev_bf16(x)
    bsf8.set_option(bsf8.OPT_GEMM_PATH, AHEAD)
    try:
        if rows:
            y = bf16_bits(bsf8.gemm_rows(x_d, w8_d, ex_d, split_k=S))
            y2 = bf16_bits(bsf8.gemm_rows(x_d, w8_d, ex_d, split_k=S))
            two = y
        else:
            y = bf16_bits(bsf8.gemm(x_d, w8_d, ex_d, split_k=S))
            y2 = bf16_bits(bsf8.gemm(x_d, w8_d, ex_d, split_k=S))
            two = bf16_bits(bsf8.splitk_reduce(bsf8.gemm_partials(x_d, w8_d, ex_d, S)))
        assert bsf8.device_status() == 0
    finally:
        bsf8.set_option(bsf8.OPT_GEMM_PATH, 0)
    assert np.array_equal(y, y2)
    assert np.array_equal(y, two)
    return y


def test_one_hot_every_code_and_exponent(bsf8_lib):
    """x rows are unit vectors, so every output is one exact product: every code under
    every exponent byte (row block b has exponent byte b) must come back bit for bit, from
    the shared-memory A columns (0..127 of a task) and the tensor-memory ones (128..)."""
    M, N, K = 8, 256 * 32, 512
    assert plan_holds(M, K, 1)
    w8 = ((np.arange(N * K) + np.arange(N * K) // K) % 256).astype(np.uint8).reshape(1, N, K)
    ex = np.repeat(np.arange(256, dtype=np.uint8).reshape(1, 256, 1), K // 32, axis=2)
    w8_d, ex_d = to_dev_u8(w8), to_dev_u8(ex)
    bsf8.set_option(bsf8.OPT_GEMM_PATH, AHEAD)
    try:
        for k0 in range(0, K, 4 * M):
            x = np.zeros((M, K), dtype=np.uint16)
            for m in range(M):
                x[m, (k0 + 4 * m + k0 // 32) % K] = 0x3F80
            y = bf16_bits(bsf8.gemm(to_dev_bf16(x), w8_d, ex_d, split_k=1))
            assert np.all(same_bits(y, oracle.gemm(x, w8, ex), zero_sign=True)), k0
        assert bsf8.device_status() == 0
    finally:
        bsf8.set_option(bsf8.OPT_GEMM_PATH, 0)


@pytest.mark.parametrize("M,G,N,K,S", [
    (1, 2, 256, 1024, 8),    # cluster 8, tasks of 128 columns
    (6, 2, 256, 1024, 1),    # one split in two tasks of 512
    (8, 2, 256, 1024, 3),    # cluster 3: rows folded 43 a block
    (5, 3, 96, 1024, 2),     # N = 96: rows 96..127 of the block are not stored
    (6, 1, 384, 576, 1),     # down_proj's K: tasks of 288 (a partial 64-column chunk)
    (6, 1, 384, 640, 5),     # cluster 5, tasks of 128
    (13, 2, 256, 1024, 7),   # cluster 7, a short last split
    (16, 1, 256, 2048, 4),   # 16 token rows, cluster 8
    (17, 1, 256, 1024, 2),   # 32-token tile, half of it zero rows
    (32, 2, 128, 1024, 8),   # full 32-token tile
    (4, 1, 256, 128, 4),     # tasks of 32 columns: 2 MMAs, fewer than the accumulators
    (4, 1, 256, 160, 4),     # splits of 64 columns: the last one is empty
    (16, 1, 256, 5120, 1),   # cluster 10 (non-portable): K = 5120 in one split
    (6, 1, 128, 6144, 1),    # cluster 12
    (3, 2, 128, 4096, 16),   # cluster 16, tasks of 256
    (20, 1, 256, 7168, 14),  # cluster 14, rows folded 10 a block (the last block 0)
])
def test_matches_oracle(bsf8_lib, M, G, N, K, S):
    assert plan_holds(M, K, S)
    r = wl.rng(1000 + 7 * M + S)
    w8 = wl.codes(r, (G, N, K))
    ex = wl.exponents(r, (G, N // 32, K // 32), 115, 127)
    x = wl.activations(r, M, G * K)
    y = run_ahead(x, w8, ex, S)
    assert_gemm_close(y, oracle.gemm(x, w8, ex), f"M={M} G={G} N={N} K={K} S={S}")


@pytest.mark.parametrize("M,S", [(1, 1), (6, 2), (20, 4)])
def test_exponent_bands(bsf8_lib, M, S):
    """Row blocks with exponent bytes in [0, 24], [115, 127] and [130, 160] (both rebuild
    forms, the two-multiply one warp by warp wherever a lane needs it): every row band
    matches the oracle at its own scale."""
    r = wl.rng(1101 + M)
    G, N, K = 1, 384, 1024
    w8 = wl.codes(r, (G, N, K))
    ex = np.empty((G, N // 32, K // 32), dtype=np.uint8)
    bands = [(0, 24), (115, 127), (130, 160)]
    for nb in range(N // 32):
        lo, hi = bands[nb % 3]
        ex[:, nb, :] = wl.exponents(r, (G, K // 32), lo, hi)
    x = wl.activations(r, M, G * K)
    assert plan_holds(M, K, S)
    y = run_ahead(x, w8, ex, S)
    ref = oracle.gemm(x, w8, ex)
    for nb in range(N // 32):
        sl = slice(32 * nb, 32 * nb + 32)
        assert_gemm_close(y[:, :, sl], ref[:, :, sl], f"band rows {nb}")


def test_nan_codes_poison_their_rows(bsf8_lib):
    """e4m3 NaN codes (0x7F / 0xFF) in the shared-memory columns, the tensor-memory ones and
    a two-multiply block: exactly the rows holding one are NaN, for every token."""
    r = wl.rng(1201)
    G, N, K, M, S = 1, 256, 1024, 6, 2
    w8 = wl.codes(r, (G, N, K))
    ex = wl.exponents(r, (G, N // 32, K // 32), 118, 122)
    ex[0, 3, 20] = 150
    sites = [(7, 3), (40, 63), (100, 64), (110, 700), (255, 1023), (96 + 5, 20 * 32 + 9)]
    for n, k in sites:
        w8[0, n, k] = 0x7F if (n % 2) else 0xFF
    x = wl.activations(r, M, K)
    assert plan_holds(M, K, S)
    y = run_ahead(x, w8, ex, S)
    ref = oracle.gemm(x, w8, ex)
    assert np.array_equal(is_nan_bits(y), is_nan_bits(ref))
    for n, _ in sites:
        assert is_nan_bits(y[:, 0, n]).all()
    keep = np.ones(N, dtype=bool)
    keep[[n for n, _ in sites]] = False
    assert_gemm_close(y[:, :, keep], ref[:, :, keep], "nan codes")


@pytest.mark.parametrize("M,S", [(1, 1), (6, 2), (16, 8), (12, 16)])
def test_rows_exponents(bsf8_lib, M, S):
    """One exponent per weight row and 32 columns ([G, N, K/32]) through the same kernel."""
    r = wl.rng(1301 + M)
    G, N, K = 2, 256, 1024
    w8 = wl.codes(r, (G, N, K))
    ex = wl.exponents(r, (G, N, K // 32), 105, 135)
    x = wl.activations(r, M, G * K)
    assert plan_holds(M, K, S)
    y = run_ahead(x, w8, ex, S, rows=True)
    assert_gemm_close(y, oracle.gemm_rows(x, w8, ex), f"rows M={M} S={S}")


@pytest.mark.parametrize("M", [2, 6, 8])
def test_wo_a_full_size_sampled(bsf8_lib, M):
    """The wo_a shape (G = 2, 1024 x 4096, split_k = 8): group 1's last 256 rows against
    the oracle."""
    wk = wl.WO_A
    w8, ex = wk.weights()
    x = wk.x(M=M)
    assert plan_holds(M, wk.K, 8)
    y = run_ahead(x, w8, ex, 8)
    n0 = wk.N - 256
    ref = oracle.gemm(np.ascontiguousarray(x[:, wk.K:]), w8[1:, n0:], ex[1:, n0 // 32:])
    assert_gemm_close(y[:, 1:, n0:], ref, f"wo_a M={M}")


@pytest.mark.parametrize("M,S", [(12, 8), (16, 1), (24, 4), (32, 8)])
def test_default_path_for_9_to_32_rows(bsf8_lib, M, S):
    """Between 9 and 32 token rows the library picks this kernel by itself where its grid
    fits one block an SM (wo_a's G = 2, 1024 x 4096 does): the default call gives the
    forced kernel's bits, needs no workspace and matches the oracle on sampled rows."""
    wk = wl.WO_A
    assert plan_holds(M, wk.K, S)
    w8, ex = wk.weights()
    x = wk.x(M=M)
    w8_d, ex_d, x_d = to_dev_u8(w8), to_dev_u8(ex), to_dev_bf16(x)
    assert bsf8.workspace_bytes(M, wk.N, wk.K, wk.G, S) == 0
    y0 = bf16_bits(bsf8.gemm(x_d, w8_d, ex_d, split_k=S))
    y7 = run_ahead(x, w8, ex, S)
    assert np.array_equal(y0, y7)
    n0 = wk.N - 128
    ref = oracle.gemm(np.ascontiguousarray(x[:, :wk.K]), w8[:1, n0:], ex[:1, n0 // 32:])
    assert_gemm_close(y0[:, :1, n0:], ref, f"default M={M} S={S}")
