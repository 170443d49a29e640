"""block_scaled_fp8_weight_gb300 -- Python binding of libbsf8 (include/bsf8.h).

A GB300 (sm_103a) library for the decode/verify/draft-size linear layer whose weight is
kept as an fp8 "twin": e4m3 codes plus one power-of-two exponent per 32x32 block, rebuilt
exactly to bf16 inside the kernel (pages "recipes/docker-images/mia-tp4/adapter/
wo_a_w8.py" and ".../shared_pad_k.py").

This module only marshals arguments: it checks dtypes and devices, takes raw device
pointers and the current CUDA stream from torch, and calls the C ABI through ctypes.
Every computation runs in the library's CUDA kernels; there is no CPU fallback, and a
missing library or a CPU tensor raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

__all__ = [
    "Bsf8Error", "load", "make_twin", "twin_or_none", "dequant", "gemm", "gemm_partials", "gemm_f32", "splitk_reduce_f32", "make_twin_rows", "dequant_rows", "gemm_rows",
    "splitk_reduce", "pad_k", "pad_x", "workspace_bytes", "auto_split", "device_status",
    "set_option", "get_option", "OPT_PDL", "OPT_WAIT_TIMEOUT_NS", "OPT_DEBUG_SKIP_LOADS",
    "OPT_GEMM_PATH", "gemm_kernel", "KERNELS", "sm_clock_sample", "prefetch_l2",
    "MAX_M", "STATUS",
]

MAX_M = 16384
OPT_PDL, OPT_WAIT_TIMEOUT_NS, OPT_DEBUG_SKIP_LOADS, OPT_GEMM_PATH = 1, 2, 3, 4
# bsf8_gemm's kernels (BSF8_KERNEL_*), the values gemm_kernel() returns and OPT_GEMM_PATH forces
KERNELS = {2: "stream", 4: "decode_ahead", 5: "tensor_core", 6: "wide", 7: "decode_ahead_tc"}
STATUS = {0: "OK", 1: "ERR_SHAPE", 2: "ERR_ALIGN", 3: "ERR_STRIDE", 4: "ERR_WORKSPACE",
          5: "ERR_NULL", 6: "ERR_CUDA", 7: "ERR_TIMEOUT", 8: "ERR_DEVICE", 9: "ERR_VALUE"}

_lock = threading.Lock()
_lib = None


class Bsf8Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        name = STATUS.get(status, str(status))
        msg = _lib.bsf8_strerror(status).decode() if _lib is not None else name
        if _lib is not None and name in ("ERR_CUDA", "ERR_DEVICE"):
            msg += f" (cudaError {_lib.bsf8_last_cuda_error()})"
        super().__init__(f"{where}: BSF8_{name}: {msg}")


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libbsf8.so (building it first if it is missing and nvcc is available)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path):
            if not build_if_missing:
                raise RuntimeError(f"libbsf8 is not built ({path}); run build.build()")
            _build.build()
        lib = ctypes.CDLL(path)
        P, I, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        sig = {
            "bsf8_strerror": (ctypes.c_char_p, [I]),
            "bsf8_version": (I, []),
            "bsf8_last_cuda_error": (I, []),
            "bsf8_make_twin": (I, [P, P, P, P, P, I, I, I, P]),
            "bsf8_dequant": (I, [P, P, P, I, I, I, P]),
            "bsf8_gemm": (I, [P, P, P, P, I, I, I, I, I, I64, P, SZ, P]),
            "bsf8_gemm_workspace_bytes": (SZ, [I, I, I, I, I]),
            "bsf8_gemm_auto_split": (I, [I, I, I, I]),
            "bsf8_gemm_kernel": (I, [I, I, I, I, I]),
            "bsf8_sm_clock_sample": (I, [P, I, P]),
            "bsf8_prefetch_l2": (I, [P, P, I, I, I, P]),
            "bsf8_gemm_static_scratch": (I, [P, P, P, P, I, I, I, I, I, I64, P]),
            "bsf8_gemm_partials": (I, [P, P, P, P, I, I, I, I, I, I64, P]),
            "bsf8_make_twin_rows": (I, [P, P, P, P, P, I, I, I, P]),
            "bsf8_dequant_rows": (I, [P, P, P, I, I, I, P]),
            "bsf8_gemm_rows_workspace_bytes": (SZ, [I, I, I, I, I]),
            "bsf8_gemm_rows": (I, [P, P, P, P, I, I, I, I, I, I64, P, SZ, P]),
            "bsf8_splitk_reduce": (I, [P, P, I, I64, P]),
            "bsf8_splitk_reduce_f32": (I, [P, P, I, I64, P]),
            "bsf8_pad_k": (I, [P, P, P, P, I, I, I, I, I, P]),
            "bsf8_pad_x": (I, [P, I64, P, I, I, I, I, P]),
            "bsf8_device_status": (I, [P, P]),
            "bsf8_set_option": (I, [I, I64]),
            "bsf8_get_option": (I64, [I]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _check(status: int, where: str):
    if status != 0:
        raise Bsf8Error(status, where)


def _torch():
    import torch
    return torch


def _stream(t):
    torch = _torch()
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _dev(t, dtype, name):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (libbsf8 has no CPU path)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _contig(t, name):
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


# ----------------------------------------------------------------------- twin

def make_twin(w):
    """bf16 W [G,N,K] (or [N,K]) -> (accepted, w8 uint8 [G,N,K], exp uint8 [G,N/32,K/32],
    block_ok uint8 [G,N/32,K/32]).  Synchronises once to read `accepted`."""
    torch = _torch()
    lib = load()
    w3 = w.unsqueeze(0) if w.dim() == 2 else w
    _contig(w3, "w")
    G, N, K = w3.shape
    w8 = torch.empty((G, N, K), dtype=torch.uint8, device=w.device)
    ex = torch.empty((G, N // 32, K // 32), dtype=torch.uint8, device=w.device)
    ok = torch.empty((G, N // 32, K // 32), dtype=torch.uint8, device=w.device)
    acc = torch.empty((1,), dtype=torch.int32, device=w.device)
    _check(lib.bsf8_make_twin(_dev(w3, torch.bfloat16, "w"), _dev(w8, torch.uint8, "w8"),
                              _dev(ex, torch.uint8, "exp"), _dev(ok, torch.uint8, "block_ok"),
                              _dev(acc, torch.int32, "accepted"), G, N, K, _stream(w3)),
           "bsf8_make_twin")
    return bool(acc.item()), w8, ex, ok


def twin_or_none(w):
    """The pages' convention: (w8, exp) if the twin reproduces w exactly, else None."""
    accepted, w8, ex, _ = make_twin(w)
    return (w8, ex) if accepted else None


def dequant(w8, ex, out=None):
    """Twin -> bf16 [G,N,K], exactly bf16(e4m3 * 2^(exp-127))."""
    torch = _torch()
    lib = load()
    _contig(w8, "w8")
    _contig(ex, "exp")
    G, N, K = w8.shape
    if out is None:
        out = torch.empty((G, N, K), dtype=torch.bfloat16, device=w8.device)
    _check(lib.bsf8_dequant(_dev(w8, torch.uint8, "w8"), _dev(ex, torch.uint8, "exp"),
                            _dev(out, torch.bfloat16, "out"), G, N, K, _stream(w8)),
           "bsf8_dequant")
    return out


# ------------------------------------------ per-(row, 32-column) scale variant

def make_twin_rows(w):
    """make_twin with one exponent per (row, 32 columns): (accepted, w8 [G,N,K],
    exp [G,N,K/32], block_ok [G,N,K/32]).  Synchronises once to read `accepted`."""
    torch = _torch()
    lib = load()
    w3 = w.unsqueeze(0) if w.dim() == 2 else w
    _contig(w3, "w")
    G, N, K = w3.shape
    w8 = torch.empty((G, N, K), dtype=torch.uint8, device=w.device)
    ex = torch.empty((G, N, K // 32), dtype=torch.uint8, device=w.device)
    ok = torch.empty((G, N, K // 32), dtype=torch.uint8, device=w.device)
    acc = torch.empty((1,), dtype=torch.int32, device=w.device)
    _check(lib.bsf8_make_twin_rows(_dev(w3, torch.bfloat16, "w"), _dev(w8, torch.uint8, "w8"),
                                   _dev(ex, torch.uint8, "exp"), _dev(ok, torch.uint8, "block_ok"),
                                   _dev(acc, torch.int32, "accepted"), G, N, K, _stream(w3)),
           "bsf8_make_twin_rows")
    return bool(acc.item()), w8, ex, ok


def dequant_rows(w8, ex, out=None):
    """Twin with per-(row, 32-column) exponents -> bf16 [G,N,K]."""
    torch = _torch()
    lib = load()
    _contig(w8, "w8")
    _contig(ex, "exp")
    G, N, K = w8.shape
    if out is None:
        out = torch.empty((G, N, K), dtype=torch.bfloat16, device=w8.device)
    _check(lib.bsf8_dequant_rows(_dev(w8, torch.uint8, "w8"), _dev(ex, torch.uint8, "exp"),
                                 _dev(out, torch.bfloat16, "out"), G, N, K, _stream(w8)),
           "bsf8_dequant_rows")
    return out


def gemm_rows(x, w8, ex, split_k: int = 0, out=None, workspace=None):
    """The GEMM with per-(row, 32-column) exponents ex [G,N,K/32]; bf16 [M,G,N]."""
    torch = _torch()
    lib = load()
    _contig(w8, "w8")
    _contig(ex, "exp")
    G, N, K = w8.shape
    M, ldx = _x_view(x, G, K)
    if out is None:
        out = torch.empty((M, G, N), dtype=torch.bfloat16, device=x.device)
    need = int(lib.bsf8_gemm_rows_workspace_bytes(M, N, K, G, split_k)) if 1 <= M <= MAX_M else 0
    ws_ptr, ws_bytes = ctypes.c_void_p(0), 0
    if need:
        if workspace is None:
            workspace = torch.empty((need,), dtype=torch.uint8, device=x.device)
        ws_ptr, ws_bytes = _dev(workspace, torch.uint8, "workspace"), workspace.numel()
    _check(lib.bsf8_gemm_rows(_dev(x, torch.bfloat16, "x"), _dev(w8, torch.uint8, "w8"),
                              _dev(ex, torch.uint8, "exp"), _dev(out, torch.bfloat16, "y"),
                              M, N, K, G, split_k, ldx, ws_ptr, ws_bytes, _stream(x)), "bsf8_gemm_rows")
    return out


# ----------------------------------------------------------------------- GEMM

def _x_view(x, G, K):
    """Accept x as [M, ldx] (2-D, unit column stride) or [M, G, K] with strides
    (>= G*K, K, 1); return (M, ldx)."""
    if x.dim() == 3:
        M = x.shape[0]
        if tuple(x.shape[1:]) != (G, K) or x.stride(2) != 1 or x.stride(1) != K:
            raise ValueError("x [M,G,K] must have strides (>=G*K, K, 1)")
        return M, x.stride(0)
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be [M, ldx] with unit column stride or [M, G, K]")
    return x.shape[0], x.stride(0)


def workspace_bytes(M, N, K, G, split_k=0) -> int:
    return int(load().bsf8_gemm_workspace_bytes(M, N, K, G, split_k))


def auto_split(M, N, K, G) -> int:
    r = load().bsf8_gemm_auto_split(M, N, K, G)
    if r < 0:
        raise Bsf8Error(-r, "bsf8_gemm_auto_split")
    return r


def gemm_kernel(M, N, K, G, split_k=0) -> int:
    """The kernel bsf8_gemm runs for these sizes (a KERNELS key); raises when a kernel forced
    through OPT_GEMM_PATH cannot run the call."""
    r = load().bsf8_gemm_kernel(M, N, K, G, split_k)
    if r < 0:
        raise Bsf8Error(-r, "bsf8_gemm_kernel")
    return r


def gemm(x, w8, ex, split_k: int = 0, out=None, workspace=None):
    """y[m,g,n] = sum_k x[m, g*K+k] * W[g,n,k] with W rebuilt from the twin; bf16 [M,G,N]."""
    torch = _torch()
    lib = load()
    _contig(w8, "w8")
    _contig(ex, "exp")
    G, N, K = w8.shape
    M, ldx = _x_view(x, G, K)
    if out is None:
        out = torch.empty((M, G, N), dtype=torch.bfloat16, device=x.device)
    need = int(lib.bsf8_gemm_workspace_bytes(M, N, K, G, split_k)) if 1 <= M <= MAX_M else 0
    ws_ptr, ws_bytes = ctypes.c_void_p(0), 0
    if need:
        if workspace is None:
            workspace = torch.empty((need,), dtype=torch.uint8, device=x.device)
        ws_ptr, ws_bytes = _dev(workspace, torch.uint8, "workspace"), workspace.numel()
    _check(lib.bsf8_gemm(_dev(x, torch.bfloat16, "x"), _dev(w8, torch.uint8, "w8"),
                         _dev(ex, torch.uint8, "exp"), _dev(out, torch.bfloat16, "y"),
                         M, N, K, G, split_k, ldx, ws_ptr, ws_bytes, _stream(x)), "bsf8_gemm")
    return out


def gemm_partials(x, w8, ex, split_k: int, out=None):
    """First pass alone: fp32 partials [S, M, G, N]."""
    torch = _torch()
    lib = load()
    G, N, K = w8.shape
    M, ldx = _x_view(x, G, K)
    if out is None:
        out = torch.empty((split_k, M, G, N), dtype=torch.float32, device=x.device)
    _check(lib.bsf8_gemm_partials(_dev(x, torch.bfloat16, "x"), _dev(w8, torch.uint8, "w8"),
                                  _dev(ex, torch.uint8, "exp"), _dev(out, torch.float32, "partials"),
                                  M, N, K, G, split_k, ldx, _stream(x)), "bsf8_gemm_partials")
    return out


def splitk_reduce(P, out=None):
    """Second pass alone: bf16( ((P[0] + P[1]) + ...) ) over the leading axis."""
    torch = _torch()
    lib = load()
    _contig(P, "partials")
    S = P.shape[0]
    count = P[0].numel()
    if out is None:
        out = torch.empty(P.shape[1:], dtype=torch.bfloat16, device=P.device)
    _check(lib.bsf8_splitk_reduce(_dev(P, torch.float32, "partials"), _dev(out, torch.bfloat16, "y"),
                                  S, count, _stream(P)), "bsf8_splitk_reduce")
    return out


def splitk_reduce_f32(P, out=None):
    """The fixed-order sum over the leading axis kept in fp32."""
    torch = _torch()
    lib = load()
    _contig(P, "partials")
    S = P.shape[0]
    count = P[0].numel()
    if out is None:
        out = torch.empty(P.shape[1:], dtype=torch.float32, device=P.device)
    _check(lib.bsf8_splitk_reduce_f32(_dev(P, torch.float32, "partials"), _dev(out, torch.float32, "y"),
                                      S, count, _stream(P)), "bsf8_splitk_reduce_f32")
    return out


def gemm_f32(x, w8, ex, split_k: int = 0):
    """The GEMM with fp32 output [M,G,N] (the head's fp32-logits variant): the partials of
    the kernel the shape selects, summed over the splits in fixed order in fp32."""
    G, N, K = w8.shape
    M, _ = _x_view(x, G, K)
    S = split_k or auto_split(M, N, K, G)
    P = gemm_partials(x, w8, ex, S)
    return P[0] if S == 1 else splitk_reduce_f32(P)


# ----------------------------------------------------------------------- L2 prefetch

def prefetch_l2(w8, ex, stream=None):
    """Pull the twin (w8 [G,N,K], ex [G,N/32,K/32]) into L2 on `stream` (default: the
    current stream); a hint that changes no result."""
    torch = _torch()
    lib = load()
    _contig(w8, "w8")
    _contig(ex, "exp")
    G, N, K = w8.shape
    s = torch.cuda.current_stream(w8.device) if stream is None else stream
    _check(lib.bsf8_prefetch_l2(_dev(w8, torch.uint8, "w8"), _dev(ex, torch.uint8, "exp"), G, N, K,
                                ctypes.c_void_p(s.cuda_stream)), "bsf8_prefetch_l2")


# ----------------------------------------------------------------------- pad-K

def pad_k(w8, ex, Kp: int, pad_exp: int = 127):
    """Twin [G,N,K] -> [G,N,Kp]: zero codes and pad_exp exponents in the new columns."""
    torch = _torch()
    lib = load()
    G, N, K = w8.shape
    wo = torch.empty((G, N, Kp), dtype=torch.uint8, device=w8.device)
    eo = torch.empty((G, N // 32, Kp // 32), dtype=torch.uint8, device=w8.device)
    _check(lib.bsf8_pad_k(_dev(w8, torch.uint8, "w8"), _dev(ex, torch.uint8, "exp"),
                          _dev(wo, torch.uint8, "w8_out"), _dev(eo, torch.uint8, "exp_out"),
                          G, N, K, Kp, pad_exp, _stream(w8)), "bsf8_pad_k")
    return wo, eo


def pad_x(x, G: int, K: int, Kp: int, out=None):
    """x [M, ldx] (group g in columns [g*K, (g+1)*K)) -> [M, G*Kp] with zero tails."""
    torch = _torch()
    lib = load()
    M, ldx = x.shape[0], x.stride(0)
    if out is None:
        out = torch.empty((M, G * Kp), dtype=torch.bfloat16, device=x.device)
    _check(lib.bsf8_pad_x(_dev(x, torch.bfloat16, "x"), ldx, _dev(out, torch.bfloat16, "x_out"),
                          M, G, K, Kp, _stream(x)), "bsf8_pad_x")
    return out


# ----------------------------------------------------------------------- status

def device_status(stream=None) -> int:
    """Synchronise the stream, read and clear the library's device status word."""
    torch = _torch()
    lib = load()
    st = ctypes.c_int(0)
    s = torch.cuda.current_stream() if stream is None else stream
    _check(lib.bsf8_device_status(ctypes.byref(st), ctypes.c_void_p(s.cuda_stream)),
           "bsf8_device_status")
    return st.value


def sm_clock_sample(out, stream=None):
    """Diagnostic: per-SM (global ns timer, cycle counter) into out, an int64 CUDA tensor
    [nsm, 2] (see bsf8_sm_clock_sample)."""
    torch = _torch()
    lib = load()
    if out.dim() != 2 or out.shape[1] != 2:
        raise ValueError("out must be [nsm, 2]")
    s = torch.cuda.current_stream(out.device) if stream is None else stream
    _check(lib.bsf8_sm_clock_sample(_dev(out, torch.int64, "out"), out.shape[0],
                                    ctypes.c_void_p(s.cuda_stream)), "bsf8_sm_clock_sample")
    return out


def set_option(option: int, value: int):
    _check(load().bsf8_set_option(option, value), "bsf8_set_option")


def get_option(option: int) -> int:
    return int(load().bsf8_get_option(option))
