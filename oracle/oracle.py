"""Python access to the fp64 CPU oracle (moe_oracle.c).

TEST INFRASTRUCTURE: only the tests, the smoke check and the benchmark's CPU
baseline leg use this module.  It never touches the CUDA library.

The C file is compiled with gcc into oracle/_build/libmoe_oracle.so on first
use (or by build()); the build is a plain `gcc -O2 -fopenmp -shared`.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_OUT_DIR, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None


class _Shape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("H", ctypes.c_int32), ("I", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32)]


def build(force: bool = False) -> str:
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
                               "-fvisibility=hidden", "-Wall", "-Wno-unknown-pragmas",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i64, i32 = ctypes.c_int64, ctypes.c_int32
            L.oracle_route.argtypes = [i64, i32, i32, P, P, P]
            L.oracle_dispatch.argtypes = [i64, i32, i32, P, P, P, P, P]
            L.oracle_forward.argtypes = [P, P, P, P, P, P, P, P, P, P, i64, P, P, P]
            L.oracle_backward_tokens.argtypes = [P, P, P, P, P, P, P, P, P, i32, P, P, P, P, P, P, i64, P, P,
                                                 P, P]
            L.oracle_dw_full.argtypes = [P, P, P, P, P, P, P, P, i32, P, P, P, P, P, P, P, P, P]
            L.oracle_dw_elements.argtypes = [P, P, P, P, P, P, P, P, i32, P, P, P, P, P, P, i64, P, P, P, P,
                                             P]
            L.oracle_expert_rows.argtypes = [P, P, P, P, P, P, P, P, i64, P, P, P, P, P, P]
            L.oracle_e4m3_encode.argtypes = [ctypes.c_double]
            L.oracle_e4m3_encode.restype = ctypes.c_uint8
            L.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
            L.oracle_e4m3_decode.restype = ctypes.c_double
            L.oracle_mx_scale_exp.argtypes = [ctypes.c_double]
            L.oracle_mx_scale_exp.restype = ctypes.c_int
            L.oracle_router_forward.argtypes = [i64, i32, i32, P, P, P]
            L.oracle_router_backward.argtypes = [i64, i32, i32, P, P, P, P, P]
            L.oracle_round_bf16.argtypes = [ctypes.c_double]
            L.oracle_round_bf16.restype = ctypes.c_double
            L.oracle_mx_quantize_rows_bf16.argtypes = [i64, i64, P, P, P, P]
            L.oracle_mx_quantize_cols_bf16.argtypes = [i64, i64, i64, P, P, P]
            for f in ("oracle_route", "oracle_dispatch", "oracle_forward", "oracle_backward_tokens",
                      "oracle_expert_rows",
                      "oracle_dw_full", "oracle_dw_elements", "oracle_mx_quantize_rows_bf16",
                      "oracle_mx_quantize_cols_bf16", "oracle_router_forward", "oracle_router_backward"):
                getattr(L, f).restype = ctypes.c_int
            _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (rc={rc})")


def _shape(s):
    return _Shape(int(s.T), int(s.H), int(s.I), int(s.E), int(s.k))


def route(logits: np.ndarray, k: int):
    """Top-k expert ids [T,k] (int32) and renormalised weights [T,k] (fp64)."""
    logits = _c(logits, np.float32)
    T, E = logits.shape
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    _check(lib().oracle_route(T, E, k, _p(logits), _p(idx), _p(w)), "route")
    return idx, w


def dispatch(topk_idx: np.ndarray, E: int):
    """counts [E], offsets [E+1], row_of_slot [T,k], slot_of_row [T*k] (all int32)."""
    topk_idx = _c(topk_idx, np.int32)
    T, k = topk_idx.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    ros = np.empty((T, k), np.int32)
    sor = np.empty(T * k, np.int32)
    _check(lib().oracle_dispatch(T, E, k, _p(topk_idx), _p(counts), _p(offsets), _p(ros), _p(sor)),
           "dispatch")
    return counts, offsets, ros, sor


def _fq(fwd_quant, fW, W_gate, W_up, W_down):
    """Pointers to the forward-quantised weights (mxfp8 mode) or three NULLs."""
    if not fwd_quant:
        return None, None, None
    return fW if fW is not None else quant_weights_fwd(W_gate, W_up, W_down)


def forward(shape, x, topk_idx, topk_w, W_gate, W_up, W_down, tokens=None, want_y=False,
            fwd_quant=False, fW=None):
    """out [n,H] fp64 for the listed tokens (all tokens by default); optionally y [n,k,H].
    fwd_quant: the mxfp8 mode's forward (both forward GEMMs' operands quantised)."""
    tokens = np.arange(shape.T, dtype=np.int64) if tokens is None else _c(tokens, np.int64)
    n = len(tokens)
    out = np.empty((n, shape.H), np.float64)
    y = np.empty((n, shape.k, shape.H), np.float64) if want_y else None
    fg, fu, fd = _fq(fwd_quant, fW, W_gate, W_up, W_down)
    sh = _shape(shape)
    _check(lib().oracle_forward(ctypes.byref(sh), _p(_c(x, np.uint16)), _p(_c(topk_idx, np.int32)),
                                _p(_c(topk_w, np.float64)), _p(_c(W_gate, np.uint16)),
                                _p(_c(W_up, np.uint16)), _p(_c(W_down, np.uint16)), _p(fg), _p(fu), _p(fd),
                                n, _p(tokens), _p(out), _p(y)), "forward")
    return (out, y) if want_y else out


def expert_rows(shape, x, W_gate, W_up, W_down, tokens, experts, fwd_quant=False, fW=None):
    """g, u, a [n,I] and y [n,H] (fp64) of expert experts[q] applied to token tokens[q]."""
    tokens = _c(tokens, np.int64)
    experts = _c(experts, np.int32)
    n = len(tokens)
    g = np.empty((n, shape.I))
    u = np.empty((n, shape.I))
    a = np.empty((n, shape.I))
    y = np.empty((n, shape.H))
    fg, fu, fd = _fq(fwd_quant, fW, W_gate, W_up, W_down)
    sh = _shape(shape)
    _check(lib().oracle_expert_rows(ctypes.byref(sh), _p(_c(x, np.uint16)), _p(_c(W_gate, np.uint16)),
                                    _p(_c(W_up, np.uint16)), _p(_c(W_down, np.uint16)), _p(fg), _p(fu),
                                    _p(fd), n, _p(tokens), _p(experts), _p(g), _p(u), _p(a), _p(y)),
           "expert_rows")
    return g, u, a, y


def quant_weights(W_gate, W_up, W_down):
    """Dequantised MXFP8 copies of the weights as the backward GEMMs see them:
    W_down along H (its last axis), W_gate/W_up along I (their last axis)."""
    res = []
    for W in (W_gate, W_up, W_down):
        W = _c(W, np.uint16)
        deq = np.empty(W.shape, np.float32)
        rows = int(np.prod(W.shape[:-1]))
        _check(lib().oracle_mx_quantize_rows_bf16(rows, W.shape[-1], _p(W), None, None, _p(deq)),
               "mx_quantize_rows")
        res.append(deq)
    return tuple(res)


def quant_weights_fwd(W_gate, W_up, W_down):
    """Dequantised MXFP8 copies of the weights as the mxfp8 forward GEMMs see
    them: W_gate/W_up along H and W_down along I (each one's middle axis, the
    forward GEMM's reduction dimension)."""
    res = []
    for W in (W_gate, W_up, W_down):
        W = _c(W, np.uint16)
        E, R, C = W.shape
        Wt = np.ascontiguousarray(W.transpose(0, 2, 1))  # [E, C, R]: the reduction axis last
        deq = np.empty(Wt.shape, np.float32)
        _check(lib().oracle_mx_quantize_rows_bf16(E * C, R, _p(Wt), None, None, _p(deq)),
               "mx_quantize_rows")
        res.append(np.ascontiguousarray(deq.transpose(0, 2, 1)))
    return tuple(res)


def backward_tokens(shape, x, logits, topk_idx, topk_w, W_gate, W_up, W_down, dy, tokens=None,
                    quant=False, qW=None, fwd_quant=False, fW=None):
    """dx [n,H], d_logits [n,E], gdot [n,k] (fp64) for the listed tokens."""
    tokens = np.arange(shape.T, dtype=np.int64) if tokens is None else _c(tokens, np.int64)
    n = len(tokens)
    dx = np.empty((n, shape.H), np.float64)
    dl = np.empty((n, shape.E), np.float64)
    gd = np.empty((n, shape.k), np.float64)
    if quant and qW is None:
        qW = quant_weights(W_gate, W_up, W_down)
    qg, qu, qd = qW if quant else (None, None, None)
    fg, fu, fd = _fq(fwd_quant, fW, W_gate, W_up, W_down)
    sh = _shape(shape)
    _check(lib().oracle_backward_tokens(
        ctypes.byref(sh), _p(_c(x, np.uint16)), _p(_c(logits, np.float32)), _p(_c(topk_idx, np.int32)),
        _p(_c(topk_w, np.float64)), _p(_c(W_gate, np.uint16)), _p(_c(W_up, np.uint16)),
        _p(_c(W_down, np.uint16)), _p(_c(dy, np.uint16)), int(bool(quant)), _p(qg), _p(qu), _p(qd),
        _p(fg), _p(fu), _p(fd), n, _p(tokens), _p(dx), _p(dl), _p(gd)), "backward_tokens")
    return dx, dl, gd


def dw_full(shape, x, topk_idx, topk_w, W_gate, W_up, W_down, dy, quant=False, qW=None,
            fwd_quant=False, fW=None):
    """dW_gate, dW_up [E,H,I] and dW_down [E,I,H] (fp64)."""
    E, H, I = shape.E, shape.H, shape.I
    dWg = np.empty((E, H, I), np.float64)
    dWu = np.empty((E, H, I), np.float64)
    dWd = np.empty((E, I, H), np.float64)
    if quant and qW is None:
        qW = quant_weights(W_gate, W_up, W_down)
    qg, qu, qd = qW if quant else (None, None, None)
    fg, fu, fd = _fq(fwd_quant, fW, W_gate, W_up, W_down)
    sh = _shape(shape)
    _check(lib().oracle_dw_full(
        ctypes.byref(sh), _p(_c(x, np.uint16)), _p(_c(topk_idx, np.int32)), _p(_c(topk_w, np.float64)),
        _p(_c(W_gate, np.uint16)), _p(_c(W_up, np.uint16)), _p(_c(W_down, np.uint16)),
        _p(_c(dy, np.uint16)), int(bool(quant)), _p(qg), _p(qu), _p(qd), _p(fg), _p(fu), _p(fd),
        _p(dWg), _p(dWu), _p(dWd)), "dw_full")
    return dWg, dWu, dWd


def dw_elements(shape, x, topk_idx, topk_w, W_gate, W_up, W_down, dy, which, e, r, c, quant=False,
                qW=None, fwd_quant=False, fW=None):
    """Selected weight-gradient elements: which 0 = dW_gate[e,r,c], 1 = dW_up[e,r,c],
    2 = dW_down[e,r,c]."""
    which, e, r, c = (_c(a, np.int32) for a in (which, e, r, c))
    val = np.empty(len(which), np.float64)
    if quant and qW is None:
        qW = quant_weights(W_gate, W_up, W_down)
    qg, qu, qd = qW if quant else (None, None, None)
    fg, fu, fd = _fq(fwd_quant, fW, W_gate, W_up, W_down)
    sh = _shape(shape)
    _check(lib().oracle_dw_elements(
        ctypes.byref(sh), _p(_c(x, np.uint16)), _p(_c(topk_idx, np.int32)), _p(_c(topk_w, np.float64)),
        _p(_c(W_gate, np.uint16)), _p(_c(W_up, np.uint16)), _p(_c(W_down, np.uint16)),
        _p(_c(dy, np.uint16)), int(bool(quant)), _p(qg), _p(qu), _p(qd), _p(fg), _p(fu), _p(fd),
        len(which), _p(which), _p(e), _p(r), _p(c), _p(val)), "dw_elements")
    return val


def e4m3_encode(v: float) -> int:
    return int(lib().oracle_e4m3_encode(float(v)))


def e4m3_decode(code: int) -> float:
    return float(lib().oracle_e4m3_decode(int(code)))


def router_forward(x, W_r):
    """logits [T,E] (fp64) = x [T,H] . W_r [H,E] (bf16 bit patterns)."""
    x = _c(x, np.uint16)
    W_r = _c(W_r, np.uint16)
    T, H = x.shape
    E = W_r.shape[1]
    out = np.empty((T, E), np.float64)
    _check(lib().oracle_router_forward(T, H, E, _p(x), _p(W_r), _p(out)), "router_forward")
    return out


def router_backward(x, W_r, d_logits):
    """dW_r [H,E] and the router's dx [T,H] (fp64) for an upstream d_logits [T,E]."""
    x = _c(x, np.uint16)
    W_r = _c(W_r, np.uint16)
    g = _c(d_logits, np.float64)
    T, H = x.shape
    E = W_r.shape[1]
    dW = np.empty((H, E), np.float64)
    dx = np.empty((T, H), np.float64)
    _check(lib().oracle_router_backward(T, H, E, _p(x), _p(W_r), _p(g), _p(dW), _p(dx)), "router_backward")
    return dW, dx


def round_bf16(v: float) -> float:
    """Nearest bf16 value (ties to even), as the fp8_bwd backward rounds its tensors."""
    return float(lib().oracle_round_bf16(float(v)))


def mx_scale_exp(amax: float) -> int:
    return int(lib().oracle_mx_scale_exp(float(amax)))


def mx_quantize_rows(a_bf16: np.ndarray):
    """E4M3 codes, E8M0 scale codes and dequantised values of bf16 rows, blocks of 32 along the row."""
    a = _c(a_bf16, np.uint16)
    rows = int(np.prod(a.shape[:-1]))
    L = a.shape[-1]
    codes = np.empty(a.shape, np.uint8)
    scales = np.empty(a.shape[:-1] + (L // 32,), np.uint8)
    deq = np.empty(a.shape, np.float32)
    _check(lib().oracle_mx_quantize_rows_bf16(rows, L, _p(a), _p(codes), _p(scales), _p(deq)),
           "mx_quantize_rows")
    return codes, scales, deq


def mx_quantize_cols(a_bf16: np.ndarray, seg: int, n: int):
    """Codes [n_pad, cols] and scales [n_pad/32, cols] of rows [seg, seg+n) quantised down columns."""
    a = _c(a_bf16, np.uint16)
    cols = a.shape[1]
    npad = (n + 31) // 32 * 32
    codes = np.empty((npad, cols), np.uint8)
    scales = np.empty((npad // 32, cols), np.uint8)
    _check(lib().oracle_mx_quantize_cols_bf16(cols, seg, n, _p(a), _p(codes), _p(scales)),
           "mx_quantize_cols")
    return codes, scales
