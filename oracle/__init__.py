"""CPU oracle for the block-scaled FP8 weight path (ctypes binding of bsf8_oracle.c).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this package.
The product library (``block_scaled_fp8_weight_gb300``) never imports it and shares no
code with it.

The C source restates the pages "recipes/docker-images/mia-tp4/adapter/wo_a_w8.py"
(make_twin, the dequant rule, the grouped small-M linear with fixed-order split-K) and
"recipes/docker-images/mia-tp4/adapter/shared_pad_k.py" (the K-padding rule); each C
function names the passage it follows.  All arrays here are numpy arrays on the host;
bf16 values travel as their uint16 bit patterns.

Every function is pinned by ``tests/test_oracle_pins.py`` (see the test docstrings for
which pin covers which function).  There is no unpinned function.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bsf8_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libbsf8_oracle.so")
# No fused multiply-add and no reassociation: every step is the binary32 (or binary64)
# operation the C source spells out.
CFLAGS = ["-O1", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
          "-fno-unsafe-math-optimizations", "-fexcess-precision=standard"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C, no GPU); returns the library path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        L = ctypes.c_long
        sig = {
            "bsfo_bf16_to_f32": (ctypes.c_float, [ctypes.c_uint16]),
            "bsfo_bf16_rne": (ctypes.c_uint16, [ctypes.c_float]),
            "bsfo_e4m3_decode": (ctypes.c_float, [ctypes.c_uint8]),
            "bsfo_e4m3_rne": (ctypes.c_uint8, [ctypes.c_float]),
            "bsfo_dequant_one": (ctypes.c_uint16, [ctypes.c_uint8, ctypes.c_uint8]),
            "bsfo_twin_exponent": (I, [ctypes.c_float]),
            "bsfo_bf16_rne_array": (None, [P, P, L]),
            "bsfo_e4m3_rne_array": (None, [P, P, L]),
            "bsfo_e4m3_decode_array": (None, [P, P, L]),
            "bsfo_twin_exponent_array": (None, [P, P, L]),
            "bsfo_dequant": (None, [P, P, P, I, I, I]),
            "bsfo_make_twin": (I, [P, P, P, P, I, I, I]),
            "bsfo_gemm": (None, [P, L, P, P, P, I, I, I, I]),
            "bsfo_gemm_f64": (None, [P, L, P, P, P, P, I, I, I, I]),
            "bsfo_split_range": (None, [I, I, I, P, P]),
            "bsfo_gemm_partials": (None, [P, L, P, P, P, I, I, I, I, I]),
            "bsfo_splitk_reduce": (None, [P, P, L, I]),
            "bsfo_pad_k": (None, [P, P, P, P, I, I, I, I, ctypes.c_uint8]),
            "bsfo_pad_x": (None, [P, L, P, I, I, I, I]),
            "bsfo_dequant_rows": (None, [P, P, P, I, I, I]),
            "bsfo_make_twin_rows": (I, [P, P, P, P, I, I, I]),
            "bsfo_gemm_rows": (None, [P, L, P, P, P, I, I, I, I]),
        }
        for name, (res, args) in sig.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def _u8(a):
    return np.ascontiguousarray(a, dtype=np.uint8)


def _u16(a):
    return np.ascontiguousarray(a, dtype=np.uint16)


# ----------------------------------------------------------------- scalar codecs

def bf16_to_f32(h: int) -> float:
    return _load().bsfo_bf16_to_f32(int(h))


def bf16_rne(f: float) -> int:
    return _load().bsfo_bf16_rne(float(np.float32(f)))


def e4m3_decode(b: int) -> float:
    return _load().bsfo_e4m3_decode(int(b))


def e4m3_rne(f: float) -> int:
    return _load().bsfo_e4m3_rne(float(np.float32(f)))


def dequant_one(q: int, e: int) -> int:
    return _load().bsfo_dequant_one(int(q), int(e))


def twin_exponent(amax: float) -> int:
    return _load().bsfo_twin_exponent(float(np.float32(amax)))


def bf16_rne_array(f: np.ndarray) -> np.ndarray:
    f = np.ascontiguousarray(f, dtype=np.float32)
    out = np.empty(f.shape, dtype=np.uint16)
    _load().bsfo_bf16_rne_array(_ptr(f), _ptr(out), f.size)
    return out


def e4m3_rne_array(f: np.ndarray) -> np.ndarray:
    f = np.ascontiguousarray(f, dtype=np.float32)
    out = np.empty(f.shape, dtype=np.uint8)
    _load().bsfo_e4m3_rne_array(_ptr(f), _ptr(out), f.size)
    return out


def e4m3_decode_array(b: np.ndarray) -> np.ndarray:
    b = _u8(b)
    out = np.empty(b.shape, dtype=np.float32)
    _load().bsfo_e4m3_decode_array(_ptr(b), _ptr(out), b.size)
    return out


def twin_exponent_array(amax: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(amax, dtype=np.float32)
    out = np.empty(a.shape, dtype=np.int32)
    _load().bsfo_twin_exponent_array(_ptr(a), _ptr(out), a.size)
    return out


# ----------------------------------------------------------------- tensor ops

def dequant(w8: np.ndarray, ex: np.ndarray) -> np.ndarray:
    """w8 uint8 [G,N,K], ex uint8 [G,N/32,K/32] -> bf16 bits uint16 [G,N,K]."""
    w8, ex = _u8(w8), _u8(ex)
    G, N, K = w8.shape
    assert ex.shape == (G, N // 32, K // 32)
    out = np.empty((G, N, K), dtype=np.uint16)
    _load().bsfo_dequant(_ptr(w8), _ptr(ex), _ptr(out), G, N, K)
    return out


def make_twin(w: np.ndarray):
    """w bf16 bits uint16 [G,N,K] -> (accepted: bool, w8 [G,N,K], ex [G,N/32,K/32], ok)."""
    w = _u16(w)
    G, N, K = w.shape
    w8 = np.empty((G, N, K), dtype=np.uint8)
    ex = np.empty((G, N // 32, K // 32), dtype=np.uint8)
    ok = np.empty((G, N // 32, K // 32), dtype=np.uint8)
    acc = _load().bsfo_make_twin(_ptr(w), _ptr(w8), _ptr(ex), _ptr(ok), G, N, K)
    return bool(acc), w8, ex, ok


def gemm(x: np.ndarray, w8: np.ndarray, ex: np.ndarray, M: int | None = None) -> np.ndarray:
    """x bf16 bits uint16 [M, ldx] (ldx >= G*K) -> y bf16 bits uint16 [M,G,N]."""
    x, w8, ex = _u16(x), _u8(w8), _u8(ex)
    G, N, K = w8.shape
    M = x.shape[0] if M is None else M
    ldx = x.shape[1]
    assert ldx >= G * K
    y = np.empty((M, G, N), dtype=np.uint16)
    _load().bsfo_gemm(_ptr(x), ldx, _ptr(w8), _ptr(ex), _ptr(y), M, N, K, G)
    return y


def dequant_rows(w8: np.ndarray, ex: np.ndarray) -> np.ndarray:
    """w8 uint8 [G,N,K], ex uint8 [G,N,K/32] (one exponent per row and 32 columns) -> bf16
    bits uint16 [G,N,K]."""
    w8, ex = _u8(w8), _u8(ex)
    G, N, K = w8.shape
    assert ex.shape == (G, N, K // 32)
    out = np.empty((G, N, K), dtype=np.uint16)
    _load().bsfo_dequant_rows(_ptr(w8), _ptr(ex), _ptr(out), G, N, K)
    return out


def make_twin_rows(w: np.ndarray):
    """make_twin with 1 x 32 blocks: (accepted, w8 [G,N,K], ex [G,N,K/32], ok [G,N,K/32])."""
    w = _u16(w)
    G, N, K = w.shape
    w8 = np.empty((G, N, K), dtype=np.uint8)
    ex = np.empty((G, N, K // 32), dtype=np.uint8)
    ok = np.empty((G, N, K // 32), dtype=np.uint8)
    acc = _load().bsfo_make_twin_rows(_ptr(w), _ptr(w8), _ptr(ex), _ptr(ok), G, N, K)
    return bool(acc), w8, ex, ok


def gemm_rows(x: np.ndarray, w8: np.ndarray, ex: np.ndarray) -> np.ndarray:
    """The GEMM with per-(row, 32-column) exponents ex [G,N,K/32]."""
    x, w8, ex = _u16(x), _u8(w8), _u8(ex)
    G, N, K = w8.shape
    M, ldx = x.shape
    assert ldx >= G * K and ex.shape == (G, N, K // 32)
    y = np.empty((M, G, N), dtype=np.uint16)
    _load().bsfo_gemm_rows(_ptr(x), ldx, _ptr(w8), _ptr(ex), _ptr(y), M, N, K, G)
    return y


def gemm_f64(x: np.ndarray, w8: np.ndarray, ex: np.ndarray):
    """Binary64 sums: returns (y64 [M,G,N] float64, sum|x*w| [M,G,N] float64)."""
    x, w8, ex = _u16(x), _u8(w8), _u8(ex)
    G, N, K = w8.shape
    M, ldx = x.shape
    y = np.empty((M, G, N), dtype=np.float64)
    a = np.empty((M, G, N), dtype=np.float64)
    _load().bsfo_gemm_f64(_ptr(x), ldx, _ptr(w8), _ptr(ex), _ptr(y), _ptr(a), M, N, K, G)
    return y, a


def split_range(K: int, S: int, s: int):
    lo, hi = ctypes.c_int(), ctypes.c_int()
    _load().bsfo_split_range(K, S, s, ctypes.byref(lo), ctypes.byref(hi))
    return lo.value, hi.value


def gemm_partials(x: np.ndarray, w8: np.ndarray, ex: np.ndarray, S: int) -> np.ndarray:
    """Per-split binary32 partials P [S,M,G,N] float32."""
    x, w8, ex = _u16(x), _u8(w8), _u8(ex)
    G, N, K = w8.shape
    M, ldx = x.shape
    P = np.empty((S, M, G, N), dtype=np.float32)
    _load().bsfo_gemm_partials(_ptr(x), ldx, _ptr(w8), _ptr(ex), _ptr(P), M, N, K, G, S)
    return P


def splitk_reduce(P: np.ndarray) -> np.ndarray:
    """P float32 [S, ...] -> bf16 bits uint16 [...], summed s = 0..S-1 in order."""
    P = np.ascontiguousarray(P, dtype=np.float32)
    S = P.shape[0]
    count = int(np.prod(P.shape[1:]))
    y = np.empty(P.shape[1:], dtype=np.uint16)
    _load().bsfo_splitk_reduce(_ptr(P), _ptr(y), count, S)
    return y


def gemm_splitk(x, w8, ex, S: int) -> np.ndarray:
    """The split-K algorithm end to end: partials, then the fixed-order reduce."""
    return splitk_reduce(gemm_partials(x, w8, ex, S))


def pad_k(w8: np.ndarray, ex: np.ndarray, Kp: int, pad_exp: int = 127):
    w8, ex = _u8(w8), _u8(ex)
    G, N, K = w8.shape
    wo = np.empty((G, N, Kp), dtype=np.uint8)
    eo = np.empty((G, N // 32, Kp // 32), dtype=np.uint8)
    _load().bsfo_pad_k(_ptr(w8), _ptr(ex), _ptr(wo), _ptr(eo), G, N, K, Kp, int(pad_exp))
    return wo, eo


def pad_x(x: np.ndarray, G: int, K: int, Kp: int) -> np.ndarray:
    x = _u16(x)
    M, ldx = x.shape
    out = np.empty((M, G * Kp), dtype=np.uint16)
    _load().bsfo_pad_x(_ptr(x), ldx, _ptr(out), M, G, K, Kp)
    return out


# ----------------------------------------------------------------- helpers

def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """Reinterpret bf16 bit patterns as float32 (exact widening)."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
