"""GPU: the K-padding rule (bit-exact against the oracle, and the GEMM output left
bitwise unchanged by padding, as the shared-expert down_proj page measured), and the
device status word (a bounded wait that runs out is reported, nothing hangs)."""
import json
import os

import numpy as np
import pytest
import torch

import block_scaled_fp8_weight_gb300 as bsf8
import oracle
from block_scaled_fp8_weight_gb300 import workloads as wl
from _helpers import bf16_bits, to_dev_bf16, to_dev_u8

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_pad_k_and_pad_x_bit_exact(bsf8_lib):
    r = wl.rng(41)
    G, N, K, Kp, M = 3, 96, 160, 256, 5
    w8 = wl.codes(r, (G, N, K))
    ex = wl.exponents(r, (G, N // 32, K // 32), 110, 130)
    x = wl.activations(r, M, G * K + 16)
    for pe in (0, 127, 200, 255):
        wo, eo = bsf8.pad_k(to_dev_u8(w8), to_dev_u8(ex), Kp, pad_exp=pe)
        wr, er = oracle.pad_k(w8, ex, Kp, pad_exp=pe)
        assert np.array_equal(wo.cpu().numpy(), wr) and np.array_equal(eo.cpu().numpy(), er)
    xo = bsf8.pad_x(to_dev_bf16(x), G, K, Kp)
    assert np.array_equal(bf16_bits(xo), oracle.pad_x(x, G, K, Kp))


def test_down_proj_padding_leaves_output_bitwise_unchanged(bsf8_lib):
    """The page's LOSSLESS check: 0 of 30720 outputs differ between K = 576 and the
    zero-padded K = 640, for pad exponents 0, 127 and 200 (here at split_k = 1, where
    padding only appends zero products to each sum)."""
    facts = json.load(open(os.path.join(GOLDEN, "pages_facts.json")))
    pk, ll = facts["pad_k"], facts["pad_k_lossless"]
    wk = wl.DOWN_PROJ
    w8, ex = wk.weights()
    x = wk.x()
    w8_d, ex_d, x_d = to_dev_u8(w8), to_dev_u8(ex), to_dev_bf16(x)
    y576 = bf16_bits(bsf8.gemm(x_d, w8_d, ex_d, split_k=1))
    assert y576.size == ll["outputs"]
    xp = bsf8.pad_x(x_d, 1, pk["K"], pk["Kp"])
    for pe in ll["pad_exps_checked"]:
        wp, ep = bsf8.pad_k(w8_d, ex_d, pk["Kp"], pad_exp=pe)
        assert list(ep.shape[1:]) == pk["scale_shape_after"]
        y640 = bf16_bits(bsf8.gemm(xp, wp, ep, split_k=1))
        assert int(np.count_nonzero(y640 != y576)) == ll["differing"]
    # With splits whose boundaries coincide over the first 576 columns the bits are kept
    # as well: 6 splits of 3 blocks (576) against 7 splits of 3 blocks (640, the seventh
    # holding only the two zero blocks).
    y6 = bf16_bits(bsf8.gemm(x_d, w8_d, ex_d, split_k=6))
    wp, ep = bsf8.pad_k(w8_d, ex_d, pk["Kp"], pad_exp=127)
    y7 = bf16_bits(bsf8.gemm(xp, wp, ep, split_k=7))
    assert np.array_equal(y6, y7)


@pytest.mark.parametrize("path,M,kernel", [(0, 4, 4), (0, 40, 5), (6, 4, 6), (7, 4, 7), (7, 20, 7)])
def test_timeout_is_reported_without_hanging(bsf8_lib, path, M, kernel):
    """With the test-only option that suppresses the weight loads, the mbarrier waits of
    the decode-ahead GEMM (path 0 at M = 4), the tensor-core GEMM (path 0 at M = 40), the
    wide-weight GEMM (path 6) and the decode-ahead tensor-core GEMM (path 7, 16- and
    32-token tiles) run out after the shortened bound; the kernel records
    BSF8_ERR_TIMEOUT, writes nothing and returns.  Normal calls work again afterwards.
    The library confirms which kernel each case runs."""
    w8, ex = wl.TINY.weights()
    x = wl.TINY.x(M=M)
    w8_d, ex_d, x_d = to_dev_u8(w8), to_dev_u8(ex), to_dev_bf16(x)
    assert bsf8.device_status() == 0
    old = bsf8.get_option(bsf8.OPT_WAIT_TIMEOUT_NS)
    y = torch.full((M, 1, 256), 7.0, dtype=torch.bfloat16, device="cuda")
    try:
        bsf8.set_option(bsf8.OPT_GEMM_PATH, path)
        bsf8.set_option(bsf8.OPT_WAIT_TIMEOUT_NS, 2_000_000)     # 2 ms
        bsf8.set_option(bsf8.OPT_DEBUG_SKIP_LOADS, 1)
        for S in (1, 4):
            assert bsf8.gemm_kernel(M, 256, 512, 1, S) == kernel
            bsf8.gemm(x_d, w8_d, ex_d, split_k=S, out=y)
            assert bsf8.device_status() == 7
            assert torch.all(y == 7.0)                            # nothing written
    finally:
        bsf8.set_option(bsf8.OPT_DEBUG_SKIP_LOADS, 0)
        bsf8.set_option(bsf8.OPT_WAIT_TIMEOUT_NS, old)
    try:
        y = bsf8.gemm(x_d, w8_d, ex_d, split_k=4)
        assert bsf8.device_status() == 0
    finally:
        bsf8.set_option(bsf8.OPT_GEMM_PATH, 0)
    y = bsf8.gemm(x_d, w8_d, ex_d, split_k=4)
    assert bsf8.device_status() == 0
    ref = oracle.gemm(x, w8, ex)
    from _helpers import assert_gemm_close
    assert_gemm_close(bf16_bits(y), ref)
