"""GPU: no kernel writes outside its outputs.  Every output of the ragged and edge cases
-- y, the fp32 partials, the padded twin and activations, make_twin's codes, exponents and
flags, dequant's bf16 weight -- is placed between 4 KiB guard regions filled with a
canary byte; after the call the guards must be unchanged and the outputs must match the
oracle.  The shapes put tiles and splits across the ends of buffers: 96 weight rows (one
and a half 64-row tiles), 193 token rows (a second 192-row token tile of one row), 9..32
token rows, and splits that end inside a 64-column step."""
import ctypes

import numpy as np
import pytest
import torch

import block_scaled_fp8_weight_gb300 as bsf8
import oracle
from block_scaled_fp8_weight_gb300 import workloads as wl
from _helpers import assert_gemm_close, bf16_bits, to_dev_bf16, to_dev_u8

pytestmark = pytest.mark.gpu

GUARD = 4096
CANARY = 0xA5


def guarded(nbytes):
    """A device byte buffer with GUARD canary bytes on both sides of an nbytes window."""
    buf = torch.full((GUARD + nbytes + GUARD,), CANARY, dtype=torch.uint8, device="cuda")
    return buf, buf[GUARD:GUARD + nbytes]


def guards_intact(buf):
    torch.cuda.synchronize()
    head = buf[:GUARD].cpu().numpy()
    tail = buf[-GUARD:].cpu().numpy()
    return bool(np.all(head == CANARY) and np.all(tail == CANARY))


def ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


GEMM_CASES = [
    # G, N, K, M, S
    (1, 96, 160, 3, 1),        # 1.5 row tiles, 5 column blocks, one split
    (1, 96, 256, 193, 2),      # a second token tile holding one row (tensor-core kernel)
    (2, 160, 544, 13, 8),      # 9..32 rows, 17 blocks in 8 splits (two empty)
    (1, 64, 576, 9, 5),        # split boundaries at 128 / 256 / ... off the 64-column steps
    (1, 96, 576, 20, 7),       # 7 splits of 96 columns: each ends inside a 64-column step
    (2, 1024, 4096, 6, 7),     # wo_a in 7 splits of 608 columns
    (1, 5120, 576, 6, 7),      # down_proj in 7 splits
    (1, 128, 1024, 32, 3),     # 32 rows, uneven splits
]


@pytest.mark.parametrize("G,N,K,M,S", GEMM_CASES)
def test_gemm_and_partials_write_only_their_outputs(bsf8_lib, G, N, K, M, S):
    r = wl.rng(7000 + G * 97 + N + K + M + S)
    w8 = wl.codes(r, (G, N, K))
    ex = wl.exponents(r, (G, N // 32, K // 32), 115, 127)
    x = wl.activations(r, M, G * K)
    w8_d, ex_d, x_d = to_dev_u8(w8), to_dev_u8(ex), to_dev_bf16(x)
    ref = oracle.gemm(x, w8, ex)

    ybuf, ywin = guarded(M * G * N * 2)
    y = ywin.view(torch.bfloat16).view(M, G, N)
    need = bsf8.workspace_bytes(M, N, K, G, S)
    wbuf, wwin = guarded(max(16, need))
    bsf8.gemm(x_d, w8_d, ex_d, split_k=S, out=y, workspace=wwin if need else None)
    assert bsf8.device_status() == 0
    assert guards_intact(ybuf), "y guards"
    assert guards_intact(wbuf), "workspace guards"
    assert_gemm_close(bf16_bits(y), ref, f"G={G} N={N} K={K} M={M} S={S}")

    pbuf, pwin = guarded(S * M * G * N * 4)
    P = pwin.view(torch.float32).view(S, M, G, N)
    bsf8.gemm_partials(x_d, w8_d, ex_d, S, out=P)
    assert bsf8.device_status() == 0
    assert guards_intact(pbuf), "partials guards"
    rbuf, rwin = guarded(M * G * N * 2)
    y2 = rwin.view(torch.bfloat16).view(M, G, N)
    bsf8.splitk_reduce(P, out=y2)
    assert guards_intact(rbuf), "reduce guards"
    assert np.array_equal(bf16_bits(y2), bf16_bits(y))


def test_twin_dequant_and_padding_write_only_their_outputs(bsf8_lib):
    lib = bsf8_lib
    G, N, K, Kp, M = 2, 96, 160, 256, 193
    r = wl.rng(77)
    w8 = wl.codes(r, (G, N, K))
    ex = wl.exponents(r, (G, N // 32, K // 32), 115, 127)
    w_bits = oracle.dequant(w8, ex)
    w_d = to_dev_bf16(w_bits)

    # make_twin: codes, exponents, block flags and the accepted flag
    cb, cw = guarded(G * N * K)
    eb, ew = guarded(G * (N // 32) * (K // 32))
    ob, ow = guarded(G * (N // 32) * (K // 32))
    ab, aw = guarded(4)
    assert lib.bsf8_make_twin(ptr(w_d), ptr(cw), ptr(ew), ptr(ow), ptr(aw), G, N, K, stream()) == 0
    for b in (cb, eb, ob, ab):
        assert guards_intact(b)
    acc, t8, tex, tok = oracle.make_twin(w_bits)
    assert int(aw.view(torch.int32).item()) == int(acc)
    assert np.array_equal(cw.cpu().numpy().reshape(G, N, K), t8)
    assert np.array_equal(ew.cpu().numpy().reshape(tex.shape), tex)

    # dequant
    db, dw = guarded(G * N * K * 2)
    bsf8.dequant(to_dev_u8(w8), to_dev_u8(ex), out=dw.view(torch.bfloat16).view(G, N, K))
    assert guards_intact(db)
    assert np.array_equal(bf16_bits(dw.view(torch.bfloat16)).reshape(G, N, K), w_bits)

    # pad-K of the twin
    pwb, pww = guarded(G * N * Kp)
    peb, pew = guarded(G * (N // 32) * (Kp // 32))
    assert lib.bsf8_pad_k(ptr(to_dev_u8(w8)), ptr(to_dev_u8(ex)), ptr(pww), ptr(pew), G, N, K, Kp, 127,
                          stream()) == 0
    assert guards_intact(pwb) and guards_intact(peb)
    w8p, exp_ = oracle.pad_k(w8, ex, Kp, 127)
    assert np.array_equal(pww.cpu().numpy().reshape(G, N, Kp), w8p)
    assert np.array_equal(pew.cpu().numpy().reshape(exp_.shape), exp_)

    # pad of the activations (193 rows, two groups)
    x = wl.activations(r, M, G * K)
    xb, xw = guarded(M * G * Kp * 2)
    bsf8.pad_x(to_dev_bf16(x), G, K, Kp, out=xw.view(torch.bfloat16).view(M, G * Kp))
    assert guards_intact(xb)
    assert np.array_equal(bf16_bits(xw.view(torch.bfloat16)).reshape(M, G * Kp), oracle.pad_x(x, G, K, Kp))
