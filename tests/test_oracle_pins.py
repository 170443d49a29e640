"""Pins for the CPU oracle: each check ties an oracle function to something other than
itself -- a library cast, a hand-derived closed form, integer arithmetic, a binary64
sum with Higham's error bound, brute force over every candidate, or a value the pages
print.  None of these tests touches a GPU.

Which pin covers which oracle function:
  bf16_rne        torch's binary32 -> bfloat16 cast over random and boundary patterns
  e4m3_decode     torch's float8_e4m3fn -> float32 cast, all 256 codes
  e4m3_rne        torch's float32 -> float8_e4m3fn cast; brute-force nearest-even search
  twin_exponent   exact integer search for every bf16 amax; the pages' binary32 formula;
                  hand-derived golden values
  dequant         hand-derived golden values; e = 127 equals torch's e4m3 -> bf16 cast;
                  scaling and sign invariants over all codes x exponents
  make_twin       round trip on generated-exact weights; recovery of the generating codes;
                  rejection of exactly the nudged blocks; per-element brute-force checks
                  of exponent, nearest-even code and acceptance on non-exact weights
  gemm / gemm_f64 one-hot x (bitwise dequant); integer data (exact, vs int64 matmul);
                  Higham's bound vs the binary64 sum; binary64 sum vs numpy's float64
                  einsum (layout, groups, row stride)
  split_range, gemm_partials, splitk_reduce
                  the pages' 512-column splits; coverage; S = 1 equals gemm; integer data;
                  hand-derived order-sensitive sums
  pad_k / pad_x   the pages' padded shapes and their lossless claim (0 of 30720 differ for
                  pad exponents 0, 127, 200)
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp8_weight_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


def _bits_to_f32(b):
    return np.asarray(b, dtype=np.uint32).view(np.float32)


def _torch_bf16_bits(f32):
    t = torch.from_numpy(np.ascontiguousarray(f32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _torch_e4m3_decode_all():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float32).numpy()


def _bf16_equal_or_both_nan(a, b):
    a = np.asarray(a, dtype=np.uint16)
    b = np.asarray(b, dtype=np.uint16)
    nan_a = ((a & 0x7FFF) > 0x7F80)
    nan_b = ((b & 0x7FFF) > 0x7F80)
    return np.where(nan_a | nan_b, nan_a & nan_b, a == b)


# ----------------------------------------------------------------------------- codecs

def test_bf16_rne_matches_torch_cast():
    r = np.random.default_rng(1)
    rand = r.integers(0, 2**32, size=2_000_000, dtype=np.uint64).astype(np.uint32)
    # Boundary patterns: exact ties (low half 0x8000), one below/above, subnormals, the
    # largest finite values and the carry into infinity.
    hi = r.integers(0, 2**16, size=20_000, dtype=np.uint64).astype(np.uint32) << 16
    ties = np.concatenate([hi | 0x8000, hi | 0x7FFF, hi | 0x8001, hi])
    special = np.array([0, 0x80000000, 1, 0x007FFFFF, 0x00800000, 0x7F7FFFFF, 0x7F7F8000,
                        0x7F7F7FFF, 0x7F800000, 0xFF800000, 0x3F808000, 0x3F818000],
                       dtype=np.uint32)
    bits = np.concatenate([rand, ties, special])
    f = _bits_to_f32(bits)
    finite = ~np.isnan(f)
    ours = oracle.bf16_rne_array(f[finite])
    ref = _torch_bf16_bits(f[finite])
    assert np.array_equal(ours, ref)
    nan_out = oracle.bf16_rne_array(f[~finite])
    assert np.all((nan_out & 0x7FFF) > 0x7F80)


def test_e4m3_decode_matches_torch_all_codes():
    ref = _torch_e4m3_decode_all()
    ours = oracle.e4m3_decode_array(np.arange(256, dtype=np.uint8))
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert set(np.nonzero(nan)[0].tolist()) == {0x7F, 0xFF}
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))  # incl. -0
    assert np.nanmax(ours) == 448.0


def _e4m3_domain_values():
    """Every binary32 value make_twin hands to the encoder, plus ties and neighbours."""
    # All finite bf16 magnitudes divided by every power of two e in [-127, 120] that can
    # be a block scale for them (|w| / 2^e <= 448).
    r = np.random.default_rng(2)
    w = oracle.bf16_bits_to_f32(np.arange(0, 0x7F80, dtype=np.uint16))
    vals = []
    with np.errstate(over="ignore"):
        for e in range(-127, 121):
            q = (w * np.float32(2.0 ** -e)).astype(np.float32)
            q = q[np.isfinite(q) & (q <= 448.0)]
            vals.append(q)
    v = np.concatenate(vals)
    # midpoints between consecutive finite e4m3 magnitudes and their binary32 neighbours
    table = np.unique(_torch_e4m3_decode_all()[:0x7F])
    mids = ((table[:-1].astype(np.float64) + table[1:]) / 2).astype(np.float32)
    up = np.nextafter(mids, np.float32(np.inf))
    dn = np.nextafter(mids, np.float32(0))
    rnd = r.uniform(0, 448, size=500_000).astype(np.float32)
    v = np.concatenate([v, mids, up, dn, rnd, table])
    v = v[v <= 448.0]
    return np.concatenate([v, -v])


def test_e4m3_rne_matches_torch_cast_on_domain():
    v = _e4m3_domain_values()
    ours = oracle.e4m3_rne_array(v)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_rne_bruteforce_nearest_even():
    """Nearest of all 254 finite codes, ties to the even mantissa, zero keeps the sign."""
    table = _torch_e4m3_decode_all()
    finite_codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.int64)
    fvals = table[finite_codes].astype(np.float64)
    r = np.random.default_rng(3)
    table_pos = np.unique(table[:0x7F])
    mids = (table_pos[:-1] + table_pos[1:]) / 2
    x = np.concatenate([r.uniform(-448, 448, 20000), r.uniform(-0.02, 0.02, 20000),
                        mids, -mids, [0.0, -0.0, 2.0**-10, -2.0**-10, 448.0, -448.0]])
    x = x.astype(np.float32)
    ours = oracle.e4m3_rne_array(x)
    for xi, got in zip(x.astype(np.float64), ours):
        d = np.abs(fvals - xi)
        best = finite_codes[d == d.min()]
        if xi == 0.0 or np.all(fvals[np.isin(finite_codes, best)] == 0.0):
            want = 0x80 if np.signbit(xi) else 0x00
        else:
            cands = [c for c in best if np.sign(table[c]) == np.sign(xi) or table[c] == 0]
            if len(cands) > 1:
                cands = [c for c in cands if (c & 1) == 0]
            want = cands[0]
            if table[want] == 0:
                want = 0x80 if np.signbit(xi) else 0x00
        assert got == want, (xi, hex(got), hex(want))


# ---------------------------------------------------------------------- twin exponent

def _exact_twin_exponent(amax: Fraction) -> int:
    """Smallest integer e with 448 * 2^e >= max(amax, 2^-126), clamped to [-127, 127]."""
    a = max(amax, Fraction(1, 2**126))
    e = -200
    while Fraction(448) * (Fraction(2) ** e) < a:
        e += 1
    return max(-127, min(127, e))


def test_twin_exponent_bruteforce_all_bf16():
    bits = np.arange(0, 0x7F80, dtype=np.uint16)          # every finite non-negative bf16
    amax = oracle.bf16_bits_to_f32(bits)
    ours = oracle.twin_exponent_array(amax)
    # Exact integer search, done per binade with Fractions (a is m * 2^k exactly).
    for b, a, e in zip(bits[::97], amax[::97], ours[::97]):
        assert e == _exact_twin_exponent(Fraction(float(a))), hex(int(b))
    # Closed form of the same search for every pattern: for a = f * 2^E with f in [1, 2),
    # e = E - 8 + (f > 1.75), from 448 = 1.75 * 2^8; floor at 2^-126; clamp [-127, 127].
    a = np.maximum(amax.astype(np.float64), 2.0**-126)
    fr, ex = np.frexp(a)                      # a = fr * 2^ex, fr in [0.5, 1)
    E = ex - 1
    f = fr * 2
    want = np.clip(E - 8 + (f > 1.75), -127, 127)
    assert np.array_equal(ours, want)
    # The pages' expression evaluated in binary32 (torch), as make_twin runs it.
    t = torch.from_numpy(amax.copy()).clamp_min(2.0**-126)
    pages = torch.ceil(torch.log2(t / 448.0)).clamp(-127, 127).to(torch.int32).numpy()
    assert np.array_equal(ours, pages)


def test_twin_exponent_golden():
    for h, byte in _golden_rows("twin_exponents.txt"):
        a = oracle.bf16_to_f32(int(h, 16))
        assert oracle.twin_exponent(a) + 127 == int(byte), h


# ---------------------------------------------------------------------------- dequant

def test_dequant_golden():
    for code, e, want in _golden_rows("dequant_values.txt"):
        got = oracle.dequant_one(int(code, 16), int(e))
        if want == "NAN":
            assert (got & 0x7FFF) > 0x7F80, (code, e, hex(got))
        else:
            assert got == int(want, 16), (code, e, hex(got), want)


def test_dequant_unit_scale_is_e4m3_to_bf16_cast():
    """At exponent byte 127 the rule reduces to the plain e4m3 -> bf16 conversion."""
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.dequant(codes.reshape(1, 1, 256).repeat(32, 1), np.full((1, 1, 8), 127, np.uint8))[0, 0]
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.bfloat16)
    ref = ref.view(torch.int16).numpy().view(np.uint16)
    assert np.all(_bf16_equal_or_both_nan(ours, ref))


def test_dequant_invariants_all_codes_all_exponents():
    codes = np.arange(256, dtype=np.uint8)
    tab = np.array([[oracle.dequant_one(c, e) for e in range(256)] for c in codes], dtype=np.uint16)
    f = oracle.bf16_bits_to_f32(tab).astype(np.float64)
    dec = _torch_e4m3_decode_all().astype(np.float64)
    for c in range(128):
        if c == 0x7F:
            assert np.all(np.isnan(f[c])) and np.all(np.isnan(f[c | 0x80]))
            continue
        # sign symmetry: the negative code gives the negated value (zero keeps its sign)
        assert np.array_equal(tab[c] ^ 0x8000, tab[c | 0x80]) or c == 0
        for e in range(256):
            exact = dec[c] * 2.0 ** (e - 127)
            if e == 255:
                # the scale 2^128 itself is +inf in binary32: 0 * inf = NaN, else inf
                assert np.isnan(f[c, e]) if c == 0 else np.isinf(f[c, e])
            elif c == 0:
                assert f[c, e] == 0.0
            elif exact >= 2.0**128 * (1 - 2.0**-9):
                assert np.isinf(f[c, e])
            elif exact >= 2.0**-126:
                # normal bf16 range: an e4m3 value has at most 4 significant bits -> exact
                assert f[c, e] == exact, (hex(c), e)
            else:
                # bf16 subnormal range: nearest multiple of 2^-133, ties to even
                q = exact / 2.0**-133
                n = np.floor(q)
                frac = q - n
                want = n + (1 if frac > 0.5 or (frac == 0.5 and n % 2 == 1) else 0)
                assert f[c, e] == want * 2.0**-133, (hex(c), e)


# -------------------------------------------------------------------------- make_twin

def _tiny_exact_weight():
    w8, ex = wl.TINY.weights()
    return w8, ex, oracle.dequant(w8, ex)


def test_make_twin_round_trip_on_exact_weights():
    w8, ex, w = _tiny_exact_weight()
    accepted, t8, tex, ok = oracle.make_twin(w)
    assert accepted and ok.all()
    back = oracle.dequant(t8, tex)
    assert np.array_equal(oracle.bf16_bits_to_f32(back), oracle.bf16_bits_to_f32(w))
    # Blocks whose generating codes reach +-448 recover the generating exponent and codes
    # bit for bit: the block maximum is then 448 * 2^(e-127), so make_twin picks that e.
    G, N, K = w8.shape
    blk_codes = w8.reshape(G, N // 32, 32, K // 32, 32).transpose(0, 1, 3, 2, 4)
    has_max = np.any((blk_codes & 0x7F) == 0x7E, axis=(3, 4))
    assert has_max.sum() > 0
    assert np.array_equal(tex[has_max], ex[has_max])
    tcodes = t8.reshape(G, N // 32, 32, K // 32, 32).transpose(0, 1, 3, 2, 4)
    assert np.array_equal(tcodes[has_max], blk_codes[has_max])


def test_make_twin_rejects_exactly_the_nudged_blocks():
    _, _, w = _tiny_exact_weight()
    G, N, K = w.shape
    sites = wl.nudge_sites(wl.rng(5), G, N, K, frac=0.01)
    assert len(sites) == max(1, round(0.01 * G * (N // 32) * (K // 32)))
    wn = wl.apply_nudge(w, sites)
    accepted, _, _, ok = oracle.make_twin(wn)
    assert not accepted
    want = np.ones_like(ok)
    for s in sites:
        g, rem = divmod(s, N * K)
        n, k = divmod(rem, K)
        want[g, n // 32, k // 32] = 0
    assert np.array_equal(ok, want)


def test_make_twin_special_blocks():
    w = np.zeros((1, 32, 96), dtype=np.uint16)
    w[0, :, 32:64] = 0x8000          # block 1: all -0
    w[0, 5, 70] = 0x43E0             # block 2: a single 448, rest +0
    accepted, t8, tex, ok = oracle.make_twin(w)
    assert accepted and ok.all()
    assert tex.tolist() == [[[0, 0, 127]]]        # zero blocks: 2^-126 floor -> e = -127
    assert np.all(t8[0, :, :32] == 0x00) and np.all(t8[0, :, 32:64] == 0x80)
    assert t8[0, 5, 70] == 0x7E
    # a single 1.0: e = -8, the code is 1.0 / 2^-8 = 256 = 0x78 (E=15, m=0)
    w1 = np.zeros((1, 32, 32), dtype=np.uint16)
    w1[0, 0, 0] = 0x3F80
    acc1, t1, e1, _ = oracle.make_twin(w1)
    assert acc1 and e1[0, 0, 0] == 119 and t1[0, 0, 0] == 0x78
    # non-finite blocks: flag 0, exponent byte 0xFF, every code 0x7F; tensor rejected
    for bad in (0x7F80, 0xFF80, 0x7FC0):
        wb = np.zeros((1, 32, 64), dtype=np.uint16)
        wb[0, 3, 40] = bad
        accb, tb, eb, okb = oracle.make_twin(wb)
        assert not accb
        assert okb.tolist() == [[[1, 0]]] and eb[0, 0, 1] == 0xFF
        assert np.all(tb[0, :, 32:] == 0x7F) and np.all(tb[0, :, :32] == 0x00)


def test_make_twin_bruteforce_on_random_weights():
    """N(0,1) weights are not exact: every element checked against brute force."""
    r = wl.rng(7)
    w = wl.activations(r, 64, 128).reshape(1, 64, 128)
    w[0, 0, :32] = wl.activations(r, 1, 32)[0] & 0x807F     # a block of tiny values
    accepted, t8, tex, ok = oracle.make_twin(w)
    wf = oracle.bf16_bits_to_f32(w).astype(np.float64)
    table = _torch_e4m3_decode_all().astype(np.float64)
    finite_codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)])
    all_ok = True
    for bi in range(2):
        for bj in range(4):
            blk = wf[0, bi * 32:(bi + 1) * 32, bj * 32:(bj + 1) * 32]
            e = _exact_twin_exponent(Fraction(float(np.abs(blk).max())))
            assert tex[0, bi, bj] == e + 127
            block_ok = True
            for rr in range(32):
                for cc in range(32):
                    v = blk[rr, cc] / 2.0**e
                    q = t8[0, bi * 32 + rr, bj * 32 + cc]
                    d = np.abs(table[finite_codes] - v)
                    assert abs(table[q] - v) == d.min()
                    if d[np.argmin(d)] != 0 and np.count_nonzero(d == d.min()) > 1:
                        assert (q & 1) == 0 or table[q] == 0
                    back = _torch_bf16_bits(np.array([table[q] * 2.0**e], dtype=np.float32))[0]
                    if oracle.bf16_to_f32(back) != blk[rr, cc]:
                        block_ok = False
            assert ok[0, bi, bj] == block_ok
            all_ok &= block_ok
    assert accepted == all_ok and not accepted


# ------------------------------------------------------------------------------- GEMM

def test_gemm_one_hot_returns_dequantised_weights():
    w8, ex = wl.TINY.weights()
    G, N, K = w8.shape
    deq = oracle.dequant(w8, ex)
    ks = [0, 1, 31, 32, 255, 511]
    x = np.zeros((len(ks), G * K), dtype=np.uint16)
    for m, k in enumerate(ks):
        x[m, k] = 0x3F80
    y = oracle.gemm(x, w8, ex)
    for m, k in enumerate(ks):
        # bit for bit, except that a -0 weight comes out as +0: the running sum starts
        # at +0 and +0 + -0 = +0
        want = np.where(deq[0, :, k] == 0x8000, np.uint16(0), deq[0, :, k])
        assert np.array_equal(y[m, 0], want)


def test_gemm_integer_data_is_exact_vs_int64_matmul():
    r = np.random.default_rng(8)
    table = _torch_e4m3_decode_all()
    int_codes = np.array([c for c in range(256) if np.isfinite(table[c])
                          and table[c] == np.round(table[c]) and abs(table[c]) <= 16], dtype=np.uint8)
    G, N, K, M = 3, 64, 256, 5
    w8 = int_codes[r.integers(0, int_codes.size, size=(G, N, K))]
    ex = np.full((G, N // 32, K // 32), 127, dtype=np.uint8)
    xi = r.integers(-2, 3, size=(M, G * K + 64))
    x = _torch_bf16_bits(xi.astype(np.float32))
    y = oracle.gemm(x, w8, ex)
    wi = table[w8].astype(np.int64)
    xg = xi[:, :G * K].reshape(M, G, K).astype(np.int64)
    ref = np.einsum("mgk,gnk->mgn", xg, wi)
    assert np.abs(ref).max() < 2**24
    assert np.array_equal(y, _torch_bf16_bits(ref.astype(np.float32)))
    for S in (1, 2, 3, 8):
        assert np.array_equal(oracle.gemm_splitk(x, w8, ex, S), y)


def test_gemm_within_higham_bound_of_binary64_sum():
    w8, ex = wl.TINY.weights()
    x = wl.TINY.x()
    y = oracle.bf16_bits_to_f32(oracle.gemm(x, w8, ex)).astype(np.float64)
    y64, absprod = oracle.gemm_f64(x, w8, ex)
    K = w8.shape[2]
    u = 2.0**-24
    gamma = (K - 1) * u / (1 - (K - 1) * u)
    bound = gamma * absprod
    assert np.all(np.abs(y - y64) <= bound + 2.0**-8 * (np.abs(y64) + bound) + 1e-300)


def test_gemm_f64_layout_matches_numpy_einsum_with_groups_and_stride():
    r = wl.rng(9)
    G, N, K, M = 3, 96, 160, 7
    w8 = wl.codes(r, (G, N, K))
    ex = wl.exponents(r, (G, N // 32, K // 32), 115, 127)
    x = wl.activations(r, M, G * K + 40)            # row stride ldx = G*K + 40
    y64, _ = oracle.gemm_f64(x, w8, ex)
    W = oracle.bf16_bits_to_f32(oracle.dequant(w8, ex)).astype(np.float64)
    X = oracle.bf16_bits_to_f32(x)[:, :G * K].reshape(M, G, K).astype(np.float64)
    ref = np.einsum("mgk,gnk->mgn", X, W)
    scale = np.einsum("mgk,gnk->mgn", np.abs(X), np.abs(W))
    assert np.all(np.abs(y64 - ref) <= 1e-12 * scale + 1e-300)
    # the binary32 oracle agrees with its binary64 sum to bf16 rounding plus the bound
    y = oracle.bf16_bits_to_f32(oracle.gemm(x, w8, ex)).astype(np.float64)
    assert np.all(np.abs(y - ref) <= (K * 2.0**-24 * 1.01) * scale + 2.0**-8 * np.abs(ref) + 1e-30)


def test_gemm_nan_and_inf_propagation():
    w8 = np.full((1, 32, 32), 0x38, dtype=np.uint8)   # all 1.0
    ex = np.full((1, 1, 1), 127, dtype=np.uint8)
    x = np.zeros((2, 32), dtype=np.uint16)
    x[0, 3] = 0x7F80                                  # +inf
    w8[0, 7, 3] = 0x00                                # 0 * inf = NaN in row 7
    y = oracle.gemm(x, w8, ex)
    assert y[0, 0, 0] == 0x7F80 and (y[0, 0, 7] & 0x7FFF) > 0x7F80
    assert np.all(y[1] == 0)
    w8[0, 9, 5] = 0x7F                                # NaN code poisons row 9
    y = oracle.gemm(x, w8, ex)
    assert (y[1, 0, 9] & 0x7FFF) > 0x7F80 and y[1, 0, 8] == 0


# ---------------------------------------------------------------------------- split-K

def test_split_ranges_follow_the_pages_and_cover_k():
    facts = json.load(open(os.path.join(GOLDEN, "pages_facts.json")))["split_k_small"]
    for s in range(facts["S"]):
        assert oracle.split_range(facts["K"], facts["S"], s) == (
            s * facts["columns_per_split"], (s + 1) * facts["columns_per_split"])
    for K in (32, 96, 576, 640, 4096, 5120):
        for S in (1, 2, 3, 4, 7, 8, 16):
            if S > K // 32:
                continue
            spans = [oracle.split_range(K, S, s) for s in range(S)]
            assert spans[0][0] == 0 and spans[-1][1] == K
            for (a, b), (c, d) in zip(spans, spans[1:]):
                assert b == c and a <= b and a % 32 == 0


def test_splitk_reduce_golden_order():
    for row in _golden_rows("splitk_order.txt"):
        arrow = row.index("->")
        P = np.array([int(v, 16) for v in row[:arrow]], dtype=np.uint32).view(np.float32)
        got = oracle.splitk_reduce(P.reshape(-1, 1))[0]
        assert got == int(row[arrow + 1], 16), row


def test_splitk_single_split_equals_gemm():
    w8, ex = wl.TINY.weights()
    x = wl.TINY.x()
    assert np.array_equal(oracle.gemm_splitk(x, w8, ex, 1), oracle.gemm(x, w8, ex))
    P = oracle.gemm_partials(x, w8, ex, 4)
    # each partial is the binary32 sum of its own column range
    for s in range(4):
        lo, hi = oracle.split_range(512, 4, s)
        xs = np.zeros_like(x)
        xs[:, lo:hi] = x[:, lo:hi]
        ref = oracle.gemm_partials(xs, w8, ex, 1)[0]
        assert np.allclose(P[s], ref, rtol=0, atol=1e-6 * np.abs(ref).max())


# ------------------------------------------------------------------------------ pad-K

def test_pad_k_shapes_and_lossless_claim_from_the_pages():
    facts = json.load(open(os.path.join(GOLDEN, "pages_facts.json")))
    pk, ll = facts["pad_k"], facts["pad_k_lossless"]
    wk = wl.DOWN_PROJ
    assert (wk.N, wk.K) == (pk["N"], pk["K"])
    w8, ex = wk.weights()
    assert list(ex.shape[1:]) == pk["scale_shape_before"]
    x = wk.x()
    assert x.shape[0] == ll["M"]
    y = oracle.gemm(x, w8, ex)
    assert y.size == ll["outputs"]
    xp = oracle.pad_x(x, 1, pk["K"], pk["Kp"])
    assert np.all(xp[:, pk["K"]:] == 0) and np.array_equal(xp[:, :pk["K"]], x)
    for pe in ll["pad_exps_checked"]:
        wp, ep = oracle.pad_k(w8, ex, pk["Kp"], pad_exp=pe)
        assert list(ep.shape[1:]) == pk["scale_shape_after"]
        assert np.all(wp[:, :, pk["K"]:] == 0) and np.all(ep[:, :, pk["K"] // 32:] == pe)
        yp = oracle.gemm(xp, wp, ep)
        assert int(np.count_nonzero(yp != y)) == ll["differing"]
    # scale 1.0 is exponent byte 127
    assert oracle.dequant_one(0x38, 127) == 0x3F80
    # Reading of the pages' "zero weight times any scale is zero": not for byte 255,
    # whose scale is +inf (0 * inf = NaN).
    wp, ep = oracle.pad_k(w8, ex, pk["Kp"], pad_exp=255)
    yp = oracle.gemm(xp, wp, ep)
    assert np.all((yp & 0x7FFF) > 0x7F80)


def test_pad_k_keeps_groups_apart():
    r = wl.rng(10)
    G, N, K, Kp, M = 3, 64, 96, 160, 4
    w8 = wl.codes(r, (G, N, K))
    ex = wl.exponents(r, (G, N // 32, K // 32), 115, 127)
    x = wl.activations(r, M, G * K)
    wp, ep = oracle.pad_k(w8, ex, Kp)
    xp = oracle.pad_x(x, G, K, Kp)
    assert np.array_equal(oracle.gemm(xp, wp, ep), oracle.gemm(x, w8, ex))
    for g in range(G):
        assert np.array_equal(xp[:, g * Kp:g * Kp + K], x[:, g * K:(g + 1) * K])
        assert np.array_equal(wp[g, :, :K], w8[g])


# ------------------------------------------------ per-(row, 32-column) scale variant

def _expand_rows(ex):
    """Block exponents [G, N/32, K/32] -> the same exponent on every row [G, N, K/32]."""
    return np.repeat(ex, 32, axis=1)


def test_dequant_rows_equals_block_dequant_with_repeated_exponents():
    """With each 32x32 block's exponent copied to its 32 rows, the per-row rebuild is the
    block rebuild (pinned exhaustively above), over all codes and the whole exponent range."""
    r = wl.rng(61)
    G, N, K = 2, 64, 256
    w8 = r.integers(0, 256, size=(G, N, K)).astype(np.uint8)
    ex = r.integers(0, 256, size=(G, N // 32, K // 32)).astype(np.uint8)
    a = oracle.dequant(w8, ex)
    b = oracle.dequant_rows(w8, _expand_rows(ex))
    assert np.array_equal(a, b)
    # and each row follows its own exponent: change one row's byte, only that row moves
    exr = _expand_rows(ex).copy()
    exr[1, 37, 3] = 120
    c = oracle.dequant_rows(w8, exr)
    diff = np.argwhere(c != b)
    assert diff.size and np.all(diff[:, 0] == 1) and np.all(diff[:, 1] == 37)
    assert np.all((diff[:, 2] >= 96) & (diff[:, 2] < 128))


def test_gemm_rows_equals_block_gemm_with_repeated_exponents():
    r = wl.rng(62)
    G, N, K, M = 2, 64, 256, 5
    w8 = wl.codes(r, (G, N, K))
    ex = wl.exponents(r, (G, N // 32, K // 32), 110, 130)
    x = wl.activations(r, M, G * K + 8)
    assert np.array_equal(oracle.gemm(x, w8, ex), oracle.gemm_rows(x, w8, _expand_rows(ex)))


def _rows_exact_weight(seed, G=1, N=64, K=128, lo=110, hi=130):
    """A bf16 weight built from codes and per-(row, 32-column) exponents, so that it has
    an exact per-row twin; every 1 x 32 segment holds a +-448 code."""
    r = wl.rng(seed)
    w8 = wl.codes(r, (G, N, K))
    w8[..., ::32] = np.where(r.integers(0, 2, size=w8[..., ::32].shape) == 1, 0xFE, 0x7E).astype(np.uint8)
    ex = wl.exponents(r, (G, N, K // 32), lo, hi)
    return w8, ex, oracle.dequant_rows(w8, ex)


def test_make_twin_rows_recovers_the_generating_twin():
    w8, ex, w = _rows_exact_weight(63)
    accepted, t8, tex, ok = oracle.make_twin_rows(w)
    assert accepted and ok.all()
    assert np.array_equal(tex, ex) and np.array_equal(t8, w8)
    assert np.array_equal(oracle.dequant_rows(t8, tex), w)


def test_make_twin_rows_exponents_against_blocks_and_brute_force():
    """On N(0,1) weights: a row segment's exponent is at most its 32x32 block's, equal in
    the rows that hold the block maximum, and each equals the exact smallest e with
    448 * 2^e >= the segment's largest magnitude."""
    r = wl.rng(64)
    w = wl.activations(r, 64, 128).reshape(1, 64, 128)
    _, _, tex_b, _ = oracle.make_twin(w)
    acc, t8, tex, ok = oracle.make_twin_rows(w)
    eb = _expand_rows(tex_b).astype(int)
    assert np.all(tex.astype(int) <= eb)
    wf = oracle.bf16_bits_to_f32(w).astype(np.float64)
    seg = np.abs(wf).reshape(1, 64, 4, 32).max(axis=3)
    blk = seg.reshape(1, 2, 32, 4).max(axis=2)
    at_max = seg == np.repeat(blk, 32, axis=1)
    assert np.array_equal(tex[at_max], eb[at_max].astype(np.uint8))
    for n in range(0, 64, 7):
        for j in range(4):
            assert tex[0, n, j] == _exact_twin_exponent(Fraction(float(seg[0, n, j]))) + 127


def test_make_twin_rows_rejects_exactly_the_nudged_segments():
    _, _, w = _rows_exact_weight(65)
    G, N, K = w.shape
    sites = [5 * K + 40, 17 * K + 3, 63 * K + 127]
    wn = wl.apply_nudge(w, sites)
    accepted, _, _, ok = oracle.make_twin_rows(wn)
    assert not accepted
    want = np.ones_like(ok)
    for s in sites:
        n, k = divmod(s, K)
        want[0, n, k // 32] = 0
    assert np.array_equal(ok, want)
