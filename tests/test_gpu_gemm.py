"""GPU parity of bsf8_gemm (and its two passes) against the CPU oracle.

Floating-point bar (the GEMM's fp32 accumulation order differs from the oracle's index
order): max |y - y_ref| <= 1e-2 * rms(y_ref) and >= 99.9% of outputs within 1 bf16 ulp.
Where the sum is exact (one-hot x, integer data) or the same fp32 operations run in the
same order (the fixed-order reduce), the bar is bit-exact.  Run-to-run results must be
bitwise identical, and the cluster (fused) reduction must equal the two-pass one.
"""
import numpy as np
import pytest
import torch

import block_scaled_fp8_weight_gb300 as bsf8
import oracle
from block_scaled_fp8_weight_gb300 import workloads as wl
from _helpers import assert_gemm_close, bf16_bits, same_bits, to_dev_bf16, to_dev_u8

pytestmark = pytest.mark.gpu


def dev(w8, ex, x):
    """Host arrays -> device tensors (w8, exp, x)."""
    return to_dev_u8(w8), to_dev_u8(ex), to_dev_bf16(x)


def run(x_d, w8_d, ex_d, S, **kw):
    return bf16_bits(bsf8.gemm(x_d, w8_d, ex_d, split_k=S, **kw))


# ---------------------------------------------------------------- exact cases

@pytest.mark.parametrize("path,M", [(0, 8), (0, 32), (0, 256), (4, 8), (5, 8), (5, 32), (5, 256),
                                    (7, 8), (7, 32)])
def test_one_hot_every_code_and_exponent(bsf8_lib, M, path):
    """x rows are unit vectors: every output is one exact product, so the GEMM must
    reproduce the oracle bit for bit (zeros by value, NaN as NaN) for all 256 codes x
    256 exponent bytes -- this checks the in-register rebuild, including subnormal
    results, scales above 2^7, the +inf scale of byte 255 and e4m3 NaN codes -- on the
    default kernel and on each forced kernel (which the library confirms it runs; the
    wide-weight kernel, which needs K in multiples of 128, has its own one-hot test)."""
    N, K = 256 * 32, 32
    w8 = (np.arange(N * K) % 256).astype(np.uint8).reshape(1, N, K)
    ex = np.arange(256, dtype=np.uint8).reshape(1, 256, 1)
    bsf8.set_option(bsf8.OPT_GEMM_PATH, path)
    try:
        if path:
            assert bsf8.gemm_kernel(M, N, K, 1, 1) == path
        for k0 in range(0, K, M):
            x = np.zeros((M, K), dtype=np.uint16)
            for m in range(M):
                x[m, (k0 + m) % K] = 0x3F80
            y = bf16_bits(bsf8.gemm(to_dev_bf16(x), to_dev_u8(w8), to_dev_u8(ex), split_k=1))
            ref = oracle.gemm(x, w8, ex)
            assert np.all(same_bits(y, ref, zero_sign=True))
    finally:
        bsf8.set_option(bsf8.OPT_GEMM_PATH, 0)


def test_integer_data_is_exact(bsf8_lib):
    """Integer weights and activations keep every partial sum exact: any order agrees."""
    r = np.random.default_rng(31)
    table = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    ints = np.array([c for c in range(256) if np.isfinite(table[c]) and table[c] == np.round(table[c])
                     and abs(table[c]) <= 16], dtype=np.uint8)
    G, N, K = 2, 160, 1024
    w8 = ints[r.integers(0, ints.size, size=(G, N, K))]
    ex = np.full((G, N // 32, K // 32), 127, dtype=np.uint8)
    for M in (1, 6, 8, 20, 40):
        xi = r.integers(-2, 3, size=(M, G * K)).astype(np.float32)
        x = torch.from_numpy(xi).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        ref = oracle.gemm(x, w8, ex)
        w8_d, ex_d, x_d = dev(w8, ex, x)
        for S in (1, 3, 8, 16):
            assert np.array_equal(run(x_d, w8_d, ex_d, S), ref), (M, S)


# ------------------------------------------------------------ tolerance cases

def check(wk, M, S, ldx_pad=0, rows=None, n_range=None, n_blocks=None, literal=False):
    w8, ex = wk.weights()
    x = wk.x(M=M)
    if ldx_pad:
        x = np.concatenate([x, np.zeros((M, ldx_pad), dtype=np.uint16)], axis=1)
    w8_d, ex_d, x_d = dev(w8, ex, x)
    y = run(x_d, w8_d, ex_d, S)
    if rows is not None:             # oracle on sampled token rows (same values there)
        y, x = y[rows], x[rows]
    if n_range is not None:          # and/or a contiguous slice of weight rows
        n0, n1 = n_range
        y = y[:, :, n0:n1]
        w8, ex = w8[:, n0:n1], ex[:, n0 // 32:n1 // 32]
    if n_blocks is not None:         # and/or whole 32-row blocks of weight rows
        b = np.asarray(n_blocks)
        n = (32 * b[:, None] + np.arange(32)[None, :]).reshape(-1)
        y = y[:, :, n]
        w8, ex = w8[:, n], ex[:, b]
    ref = oracle.gemm(x, w8, ex)
    return assert_gemm_close(y, ref, f"{wk.name} M={M} S={S}", literal=literal)


@pytest.mark.parametrize("S", [0, 1, 4])
def test_tiny(bsf8_lib, S):
    check(wl.TINY, 4, S)


@pytest.mark.parametrize("M", wl.WO_A_ROWS)
def test_wo_a_full_size(bsf8_lib, M):
    """The whole wo_a layer (12 288 outputs at M = 6): the modified tolerance and the
    literal bound max |y - y_ref| <= 1e-2 rms over every output."""
    check(wl.WO_A, M, 8, literal=True)


@pytest.mark.parametrize("S", [0, 1, 2, 8])
def test_down_proj(bsf8_lib, S):
    """The whole shared-expert down_proj (30 720 outputs), literal bound included."""
    check(wl.DOWN_PROJ, 6, S, literal=True)


@pytest.mark.parametrize("M", wl.MID_ROWS)
@pytest.mark.parametrize("S", wl.MID_SPLITS)
def test_mid_rows_sampled(bsf8_lib, M, S):
    rows = sorted({0, M // 3, M // 2, M - 1})
    check(wl.MID, M, S, rows=rows)


@pytest.mark.parametrize("M", wl.SWEEP_ROWS)
def test_gate_up_sweep(bsf8_lib, M):
    rows = sorted({0, M // 2, M - 1})
    check(wl.GATE_UP, M, 0, rows=rows)


@pytest.mark.parametrize("M", [1, 3, 6, 8, 12, 16, 128])
def test_head_sweep_sampled(bsf8_lib, M):
    """The head-like weight across the kernels' row ranges (wide-weight up to 8 rows):
    three token rows against the oracle on 64 blocks of 32 weight rows spread evenly over
    all 1024 (so that every SM's share of the rows is sampled) and on the last 2048 rows."""
    rows = sorted({0, M // 2, M - 1})
    check(wl.HEAD, M, 0, rows=rows, n_blocks=np.linspace(0, 1023, 64).round().astype(int))
    check(wl.HEAD, M, 0, rows=rows, n_range=(32768 - 2048, 32768))


@pytest.mark.parametrize("G,N,K,M,S,pad", [
    (1, 32, 32, 1, 1, 0),          # one block
    (1, 96, 96, 3, 1, 0),          # ragged row tile (64 + 32) and column stage
    (3, 96, 160, 7, 2, 8),         # three groups, row stride > G*K
    (2, 160, 544, 13, 8, 0),       # 17 blocks in 8 splits: chunk 3, two empty splits
    (1, 64, 576, 33, 5, 24),       # two token chunks of 32
    (1, 64, 1024, 9, 32, 0),       # one block per split: a cluster of 4 blocks
    (2, 128, 2048, 5, 12, 0),      # uneven splits
    (1, 64, 2560, 9, 80, 0),       # 80 tasks per slab: partials + reduce (workspace)
    (1, 96, 65536 // 8, 2, 1, 0),  # a long single split: 8 tasks of 1024 columns
    (1, 4096, 64, 192, 2, 0),      # the largest M
    (1, 256, 544, 40, 8, 0),       # tensor-core tiles: 96-column splits, the last two empty
])
def test_ragged_and_edge_shapes(bsf8_lib, G, N, K, M, S, pad):
    r = wl.rng(G * 1000 + N + K + M + S)
    w8 = wl.codes(r, (G, N, K))
    ex = wl.exponents(r, (G, N // 32, K // 32), 115, 127)
    x = wl.activations(r, M, G * K + pad)
    y = bf16_bits(bsf8.gemm(to_dev_bf16(x), to_dev_u8(w8), to_dev_u8(ex), split_k=S))
    assert_gemm_close(y, oracle.gemm(x, w8, ex), f"G={G} N={N} K={K} M={M} S={S}")


def test_zero_activations_give_positive_zero(bsf8_lib):
    w8, ex = wl.TINY.weights()
    x = np.zeros((5, 512), dtype=np.uint16)
    x[1] = 0x8000                                     # -0 activations
    y = bf16_bits(bsf8.gemm(to_dev_bf16(x), to_dev_u8(w8), to_dev_u8(ex), split_k=4))
    assert np.all(y == 0)


# ------------------------------------------------- split-K passes, determinism

@pytest.mark.parametrize("wk,M,S", [(wl.WO_A, 6, 8), (wl.TINY, 4, 4), (wl.MID, 64, 4),
                                    (wl.DOWN_PROJ, 6, 5)])
def test_fused_equals_two_pass_and_reduce_is_bit_exact(bsf8_lib, wk, M, S):
    w8, ex = wk.weights()
    x = wk.x(M=M)
    w8_d, ex_d, x_d = dev(w8, ex, x)
    fused = run(x_d, w8_d, ex_d, S)
    P = bsf8.gemm_partials(x_d, w8_d, ex_d, S)
    two = bf16_bits(bsf8.splitk_reduce(P))
    assert np.array_equal(fused, two)
    # the second pass is fp32 adds in a fixed order: bit-exact against the oracle's
    P_h = P.cpu().numpy()
    assert np.array_equal(two, oracle.splitk_reduce(P_h))
    # each partial is its split's sum (tolerance: accumulation order inside a split)
    rows = [0, M - 1]
    P_ref = oracle.gemm_partials(x[rows], w8, ex, S)
    for s in range(S):
        got = P_h[s][rows]
        ref = P_ref[s]
        scale = np.sqrt(np.mean(ref.astype(np.float64) ** 2)) + 1e-30
        assert np.max(np.abs(got - ref)) <= 1e-4 * scale * np.sqrt(wk.K)


@pytest.mark.parametrize("wk,M,S", [(wl.WO_A, 6, 8), (wl.MID, 16, 1), (wl.MID, 16, 2),
                                    (wl.MID, 96, 4), (wl.MID, 32, 8), (wl.MID, 9, 16)])
def test_run_to_run_bitwise_determinism(bsf8_lib, wk, M, S):
    w8, ex = wk.weights()
    x = wk.x(M=M)
    w8_d, ex_d, x_d = dev(w8, ex, x)
    first = run(x_d, w8_d, ex_d, S)
    for _ in range(10):
        assert np.array_equal(run(x_d, w8_d, ex_d, S), first)


def test_pdl_off_gives_the_same_bits(bsf8_lib):
    w8, ex = wl.WO_A.weights()
    x = wl.WO_A.x()
    w8_d, ex_d, x_d = dev(w8, ex, x)
    on = run(x_d, w8_d, ex_d, 8)
    bsf8.set_option(bsf8.OPT_PDL, 0)
    try:
        off = run(x_d, w8_d, ex_d, 8)
    finally:
        bsf8.set_option(bsf8.OPT_PDL, 1)
    assert np.array_equal(on, off)


def test_cuda_graph_replay_of_layer_sequence(bsf8_lib):
    """43 layers' calls captured in one CUDA graph (as the bench runs them) give the
    same bits as eager calls."""
    wk = wl.WO_A
    layers = []
    for c in range(4):
        w8, ex = wk.weights(copy=c)
        layers.append((to_dev_u8(w8), to_dev_u8(ex), to_dev_bf16(wk.x(copy=c))))
    eager = [bsf8.gemm(x, w8, ex, split_k=8) for (w8, ex, x) in layers]
    torch.cuda.synchronize()
    outs = [torch.empty_like(e) for e in eager]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for (w8, ex, x), o in zip(layers, outs):
                bsf8.gemm(x, w8, ex, split_k=8, out=o)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for e, o in zip(eager, outs):
        assert torch.equal(e.view(torch.int16), o.view(torch.int16))


def test_sequence_of_calls_matches_oracle(bsf8_lib):
    """Back-to-back calls on one stream (programmatic dependent launch overlaps them)
    each match the oracle: the next call's early weight prefetch never reads stale x."""
    wk = wl.TINY
    w8, ex = wk.weights()
    w8_d, ex_d = to_dev_u8(w8), to_dev_u8(ex)
    xs = [wk.x(copy=c) for c in range(6)]
    x_d = [to_dev_bf16(x) for x in xs]
    # chain: each call's input is written by the kernel right before it
    ys = []
    buf = torch.empty_like(x_d[0])
    for x in x_d:
        buf.copy_(x)
        ys.append(bsf8.gemm(buf, w8_d, ex_d, split_k=4))
    for x, y in zip(xs, ys):
        assert np.array_equal(bf16_bits(y), bf16_bits(bsf8.gemm(to_dev_bf16(x), w8_d, ex_d, split_k=4)))
        assert_gemm_close(bf16_bits(y), oracle.gemm(x, w8, ex))


FORCED_CASES = [("wo_a", 6, 8), ("tiny", 4, 1), ("down_proj", 6, 4), ("tiny", 3, 16), ("wo_a", 1, 80),
                ("down_proj", 6, 7)]
# (kernel, case) pairs the forced kernel cannot run: the wide-weight kernel needs K and the
# split's columns in multiples of 128, the decode-ahead tensor-core kernel at most 16 tasks
# a 128-row block
NOT_APPLICABLE = {(6, ("down_proj", 6, 4)), (6, ("tiny", 3, 16)), (6, ("wo_a", 1, 80)),
                  (6, ("down_proj", 6, 7)), (7, ("wo_a", 1, 80))}


@pytest.mark.parametrize("path", [2, 4, 5, 6, 7])
@pytest.mark.parametrize("case", FORCED_CASES)
def test_forced_kernels_match_oracle_and_each_other(bsf8_lib, path, case):
    """Each kernel forced through BSF8_OPT_GEMM_PATH (2: streaming, 4: decode-ahead, 5:
    tensor-core, 6: wide-weight, 7: decode-ahead tensor-core) in its in-block, cluster
    (S = 16) and partials (S = 80) modes, and with splits that end inside a 64-column step
    (K = 576, S = 7).  The library reports that it runs the forced kernel (or refuses the
    call with BSF8_ERR_VALUE exactly where that kernel cannot run it); the result is within
    the tolerance of the oracle, bitwise equal to its own two-pass form, and bitwise
    reproducible."""
    name, M, S = case
    wk = {"wo_a": wl.WO_A, "tiny": wl.TINY, "down_proj": wl.DOWN_PROJ}[name]
    w8, ex = wk.weights()
    x = wk.x(M=M)
    w8_d, ex_d, x_d = dev(w8, ex, x)
    bsf8.set_option(bsf8.OPT_GEMM_PATH, path)
    try:
        if (path, case) in NOT_APPLICABLE:
            with pytest.raises(bsf8.Bsf8Error) as e1:
                bsf8.gemm_kernel(M, wk.N, wk.K, wk.G, S)
            with pytest.raises(bsf8.Bsf8Error) as e2:
                bsf8.gemm(x_d, w8_d, ex_d, split_k=S)
            with pytest.raises(bsf8.Bsf8Error) as e3:
                bsf8.gemm_partials(x_d, w8_d, ex_d, S)
            assert e1.value.status == e2.value.status == e3.value.status == 9  # BSF8_ERR_VALUE
            return
        assert bsf8.gemm_kernel(M, wk.N, wk.K, wk.G, S) == path
        y = run(x_d, w8_d, ex_d, S)
        y2 = run(x_d, w8_d, ex_d, S)
        two = bf16_bits(bsf8.splitk_reduce(bsf8.gemm_partials(x_d, w8_d, ex_d, S)))
        assert bsf8.device_status() == 0
    finally:
        bsf8.set_option(bsf8.OPT_GEMM_PATH, 0)
    assert np.array_equal(y, y2)
    assert np.array_equal(y, two)
    assert_gemm_close(y, oracle.gemm(x, w8, ex))


@pytest.mark.parametrize("wk,M,S", [(wl.DOWN_PROJ, 6, 4), (wl.DOWN_PROJ, 6, 0), (wl.WO_A, 6, 8),
                                    (wl.WO_A, 2, 0), (wl.GATE_UP, 6, 0), (wl.GATE_UP, 16, 0),
                                    (wl.MID, 12, 8), (wl.MID, 64, 0), (wl.TINY, 4, 4)])
def test_default_kernel_fused_equals_partials_and_reduce(bsf8_lib, wk, M, S):
    """bsf8_gemm and bsf8_gemm_partials + bsf8_splitk_reduce run the same kernel for the
    same sizes and split count, whichever the library picks, so they give the same bits
    (down_proj at S = 4 once ran a different kernel for its partials)."""
    w8, ex = wk.weights()
    x = wk.x(M=M)
    w8_d, ex_d, x_d = dev(w8, ex, x)
    S_used = S or bsf8.auto_split(M, wk.N, wk.K, wk.G)
    fused = run(x_d, w8_d, ex_d, S)
    two = bf16_bits(bsf8.splitk_reduce(bsf8.gemm_partials(x_d, w8_d, ex_d, S_used)))
    assert bsf8.device_status() == 0
    assert np.array_equal(fused, two)
    assert bsf8.gemm_kernel(M, wk.N, wk.K, wk.G, S) == bsf8.gemm_kernel(M, wk.N, wk.K, wk.G, S_used)


@pytest.mark.parametrize("G,N,K,M,S", [
    (2, 160, 544, 40, 4),     # a 32-row last row block, a 32-column tail step, 8 padded tokens
    (1, 8192, 1024, 200, 2),  # two token tiles (192 + 8), 256 blocks: more than one wave, partials
    (3, 256, 2048, 192, 8),   # eight splits summed in one cluster
])
def test_tensor_core_split_fold_edges(bsf8_lib, G, N, K, M, S):
    """The tensor-core kernel's in-cluster split sum (one-wave calls of 2..8 splits) on
    ragged shapes, and the partials it leaves to the reduce pass otherwise: within the
    oracle's tolerance and bitwise equal to bsf8_gemm_partials + bsf8_splitk_reduce."""
    r = wl.rng(G * 7919 + N + K + M + S)
    w8 = wl.codes(r, (G, N, K))
    ex = wl.exponents(r, (G, N // 32, K // 32), 115, 127)
    x = wl.activations(r, M, G * K)
    w8_d, ex_d, x_d = dev(w8, ex, x)
    assert bsf8.gemm_kernel(M, N, K, G, S) == 5
    y = run(x_d, w8_d, ex_d, S)
    two = bf16_bits(bsf8.splitk_reduce(bsf8.gemm_partials(x_d, w8_d, ex_d, S)))
    assert bsf8.device_status() == 0
    assert np.array_equal(y, two)
    rows = sorted({0, M // 2, M - 1})
    assert_gemm_close(y[rows], oracle.gemm(x[rows], w8, ex), f"G={G} N={N} K={K} M={M} S={S}")


def test_tensor_core_fold_output_alignment(bsf8_lib):
    """y 2 bytes past an 8-byte boundary: the fold's stores take their scalar form and the
    bits are those of an aligned y."""
    wk, M, S = wl.MID, 64, 4
    w8, ex = wk.weights()
    x = wk.x(M=M)
    w8_d, ex_d, x_d = dev(w8, ex, x)
    n = M * wk.G * wk.N
    buf = torch.empty(n + 4, dtype=torch.bfloat16, device="cuda")
    y_odd = buf[1:n + 1].view(M, wk.G, wk.N)
    assert y_odd.data_ptr() % 8 == 2
    bsf8.gemm(x_d, w8_d, ex_d, split_k=S, out=y_odd)
    ref = run(x_d, w8_d, ex_d, S)
    assert bsf8.device_status() == 0
    assert np.array_equal(bf16_bits(y_odd), ref)


@pytest.mark.parametrize("M", [9, 16, 32, 64, 96, 128, 192])
@pytest.mark.parametrize("S", [1, 2, 4])
def test_tensor_core_kernel_mid_rows(bsf8_lib, M, S):
    """The tensor-core kernel on the mid-row workload (G = 4 groups of W[1024, 4096]):
    sampled token rows within the oracle's tolerance, the fused call bitwise equal to its
    two-pass form, and run-to-run bitwise reproducible.  Where two A slots (64 columns
    each) and a split's accumulators (one a run of 8 steps past 16 tokens, of 4 or 8 up to
    16, x the token tile, rows rounded up to 16) do not fit tensor memory's 512 columns --
    one split of K = 4096 past 96 rows -- the forced kernel refuses the call
    (BSF8_ERR_VALUE)."""
    wk = wl.MID
    w8, ex = wk.weights()
    x = wk.x(M=M)
    w8_d, ex_d, x_d = dev(w8, ex, x)
    bsf8.set_option(bsf8.OPT_GEMM_PATH, 5)
    try:
        steps, ntok = 4096 // S // 128, (M + 15) // 16 * 16
        fits = any(2 * 64 + (steps + run - 1) // run * ntok <= 512 for run in (4, 8))
        if not fits:
            with pytest.raises(bsf8.Bsf8Error) as e:
                bsf8.gemm(x_d, w8_d, ex_d, split_k=S)
            assert e.value.status == 9
            return
        assert bsf8.gemm_kernel(M, wk.N, wk.K, wk.G, S) == 5
        y = run(x_d, w8_d, ex_d, S)
        y2 = run(x_d, w8_d, ex_d, S)
        two = bf16_bits(bsf8.splitk_reduce(bsf8.gemm_partials(x_d, w8_d, ex_d, S)))
        assert bsf8.device_status() == 0
    finally:
        bsf8.set_option(bsf8.OPT_GEMM_PATH, 0)
    assert np.array_equal(y, y2)
    assert np.array_equal(y, two)
    rows = sorted({0, M // 2, M - 1})
    assert_gemm_close(y[rows], oracle.gemm(x[rows], w8, ex))


@pytest.mark.parametrize("M,S", [(193, 0), (256, 4), (1024, 0)])
def test_large_m_token_tiles(bsf8_lib, M, S):
    """Past 192 rows (prefill-sized calls) the tensor-core kernel takes the tokens in tiles
    of 192 (a grid index each): the mid-row weight (G = 4 groups of W[1024, 4096]) with the
    last tile partly filled, sampled token rows within the oracle's tolerance, the fused
    call bitwise equal to its two-pass form and run-to-run reproducible."""
    wk = wl.MID
    w8, ex = wk.weights()
    x = wk.x(M=M)
    w8_d, ex_d, x_d = dev(w8, ex, x)
    S_used = S or bsf8.auto_split(M, wk.N, wk.K, wk.G)
    y = run(x_d, w8_d, ex_d, S)
    y2 = run(x_d, w8_d, ex_d, S)
    two = bf16_bits(bsf8.splitk_reduce(bsf8.gemm_partials(x_d, w8_d, ex_d, S_used)))
    assert bsf8.device_status() == 0
    assert np.array_equal(y, y2)
    assert np.array_equal(y, two)
    rows = sorted({0, 191, 192, M // 2, M - 1})
    assert_gemm_close(y[rows], oracle.gemm(x[rows], w8, ex), f"mid M={M}")


def test_large_m_head_with_row_stride(bsf8_lib):
    """The head-like weight (N = 32768, K = 5120) at 512 token rows with padded x rows:
    two token rows and the last 2048 weight rows against the oracle."""
    check(wl.HEAD, 512, 0, ldx_pad=64, rows=[0, 511], n_range=(32768 - 2048, 32768))


@pytest.mark.parametrize("M,S", [(6, 0), (64, 0), (128, 2)])
def test_fp32_output_head_variant(bsf8_lib, M, S):
    """fp32 logits (the draft head's variant) on the head-like weight: against the exact
    (binary64) sums of the same products, within the worst-case error of any fp32
    summation order, |y - y64| <= K * 2^-23 * sum|x*w| (each product is exact in fp32);
    and the bf16 GEMM is these sums rounded once."""
    wk = wl.HEAD
    w8, ex = wk.weights()
    x = wk.x(M=M)
    w8_d, ex_d, x_d = dev(w8, ex, x)
    y32 = bsf8.gemm_f32(x_d, w8_d, ex_d, split_k=S).cpu().numpy()
    assert y32.dtype == np.float32 and y32.shape == (M, 1, wk.N)
    n0 = wk.N - 1024
    rows = sorted({0, M - 1})
    y64, a64 = oracle.gemm_f64(x[rows], w8[:, n0:], ex[:, n0 // 32:])
    err = np.abs(y32[rows][:, :, n0:].astype(np.float64) - y64)
    assert np.all(err <= wk.K * 2.0 ** -23 * a64)
    S_used = S or bsf8.auto_split(M, wk.N, wk.K, wk.G)
    yb = bf16_bits(bsf8.gemm(x_d, w8_d, ex_d, split_k=S_used))
    yr = torch.from_numpy(y32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(yb, yr)
