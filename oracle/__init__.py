"""CPU oracle for block-quantized integer GEMM/GEMV -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its binding) never calls it.

The arithmetic lives in ``qoracle.c`` (plain C, built with gcc
``-O2 -ffp-contract=off``); this module only builds it and marshals numpy
arrays.  Each function names the passage it follows in the C source.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qoracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

GROUP = 32


def build(force: bool = False) -> str:
    """Compile qoracle.c into liboracle.so (OpenMP if the compiler has it)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
            "-fPIC", "-shared", _SRC, "-o", _LIB + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _L():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            I32 = ctypes.c_int32
            lib.orc_num_threads.restype = ctypes.c_int
            lib.orc_f32_to_f16.restype = ctypes.c_uint16
            lib.orc_f32_to_f16.argtypes = [ctypes.c_float]
            lib.orc_f16_to_f32.restype = ctypes.c_float
            lib.orc_f16_to_f32.argtypes = [ctypes.c_uint16]
            lib.orc_quantize_act_q8.argtypes = [P, I64, I64, I64, P, P]
            lib.orc_quantize_w_q8_0.argtypes = [P, I64, I64, P, P]
            lib.orc_quantize_w_q4_0.argtypes = [P, I64, I64, P, P]
            lib.orc_group_dots.argtypes = [P, I64, I64, I64, P, ctypes.c_int, P]
            lib.orc_qgemm.argtypes = [P, P, I64, I64, I64, P, ctypes.c_int, P, P, I64, P]
            lib.orc_qgemm_rows.argtypes = [P, P, P, I64, I64, I64, P, ctypes.c_int, P, P, P]
            lib.orc_moe_route.restype = I64
            lib.orc_moe_route.argtypes = [P, I64, I32, I32, P, P, P]
            lib.orc_grouped_qgemm_moe.restype = I64
            lib.orc_grouped_qgemm_moe.argtypes = [P, P, I64, P, I64, I32, I32, P, P, I32, I64, P, P]
            lib.orc_silu_mul.argtypes = [P, I64, I64, I64, P]
            lib.orc_import_gguf.argtypes = [P, I64, I64, ctypes.c_int, P, P]
            lib.orc_splitk_merge.argtypes = [P, P, P, I32, I64, I64, P, P, P]
            lib.orc_kv3_codebook.argtypes = [P, P]
            lib.orc_wht.argtypes = [P, I64, ctypes.c_int, P]
            lib.orc_kv3_encode.argtypes = [P, I64, ctypes.c_int, P, P, P, P]
            lib.orc_kv3_decode.argtypes = [P, P, I64, ctypes.c_int, P, P]
            lib.orc_moe_combine.argtypes = [P, P, I64, I32, I64, P, P]
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return int(_L().orc_num_threads())


def f32_to_f16_bits(values) -> np.ndarray:
    """binary32 -> binary16 bit patterns, round to nearest even (qoracle.c)."""
    v = np.asarray(values, dtype=np.float32).ravel()
    f = _L().orc_f32_to_f16
    return np.array([f(float(t)) for t in v], dtype=np.uint16)


def f16_bits_to_f32(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).ravel()
    f = _L().orc_f16_to_f32
    return np.array([f(int(t)) for t in b], dtype=np.float32)


def quantize_act_q8(x: np.ndarray):
    """Activation rows -> (qx int8 [M,K], dx float32 [M,K/32]); d = max|x|/127."""
    x = _c(x, np.float32)
    M, K = x.shape
    assert K % GROUP == 0
    qx = np.empty((M, K), np.int8)
    dx = np.empty((M, K // GROUP), np.float32)
    _L().orc_quantize_act_q8(_p(x), M, K, K, _p(qx), _p(dx))
    return qx, dx


def quantize_w_q8_0(w: np.ndarray):
    """Weights [N,K] -> (qw int8 [N,K], dw binary16 bits uint16 [N,K/32])."""
    w = _c(w, np.float32)
    N, K = w.shape
    assert K % GROUP == 0
    qw = np.empty((N, K), np.int8)
    dw = np.empty((N, K // GROUP), np.uint16)
    _L().orc_quantize_w_q8_0(_p(w), N, K, _p(qw), _p(dw))
    return qw, dw


def quantize_w_q4_0(w: np.ndarray):
    """Weights [N,K] -> (qw4 uint8 [N,K/2], dw binary16 bits uint16 [N,K/32])."""
    w = _c(w, np.float32)
    N, K = w.shape
    assert K % GROUP == 0
    qw4 = np.empty((N, K // 2), np.uint8)
    dw = np.empty((N, K // GROUP), np.uint16)
    _L().orc_quantize_w_q4_0(_p(w), N, K, _p(qw4), _p(dw))
    return qw4, dw


def group_dots(qx: np.ndarray, qw: np.ndarray, K: int, wbits: int) -> np.ndarray:
    """S int32 [M,N,K/32] = per-group integer dot products."""
    qx = _c(qx, np.int8)
    qw = _c(qw, np.int8 if wbits == 8 else np.uint8)
    M, N = qx.shape[0], qw.shape[0]
    S = np.empty((M, N, K // GROUP), np.int32)
    _L().orc_group_dots(_p(qx), M, N, K, _p(qw), wbits, _p(S))
    return S


def qgemm(qx, dx, qw, dw, wbits: int, want_mag: bool = True):
    """y float32 [M,N] = sum_g dw*dx*S (binary64 sum), and mag = sum_g |dw*dx*S|."""
    qx = _c(qx, np.int8)
    dx = _c(dx, np.float32)
    qw = _c(qw, np.int8 if wbits == 8 else np.uint8)
    dw = _c(dw, np.uint16)
    M, K = qx.shape
    N = qw.shape[0]
    y = np.empty((M, N), np.float32)
    mag = np.empty((M, N), np.float64) if want_mag else None
    _L().orc_qgemm(_p(qx), _p(dx), M, N, K, _p(qw), wbits, _p(dw), _p(y), N,
                   _p(mag) if want_mag else None)
    return y, mag


def qgemm_rows(qx, dx, rows, qw, dw, wbits: int):
    """qgemm restricted to activation rows ``rows`` (output row i = rows[i])."""
    qx = _c(qx, np.int8)
    dx = _c(dx, np.float32)
    rows = _c(rows, np.int64)
    qw = _c(qw, np.int8 if wbits == 8 else np.uint8)
    dw = _c(dw, np.uint16)
    K = qx.shape[1]
    N = qw.shape[0]
    R = rows.shape[0]
    y = np.empty((R, N), np.float32)
    mag = np.empty((R, N), np.float64)
    _L().orc_qgemm_rows(_p(qx), _p(dx), _p(rows), R, N, K, _p(qw), wbits, _p(dw),
                        _p(y), _p(mag))
    return y, mag


def moe_route(topk_ids: np.ndarray, E: int):
    """(counts [E], offsets [E+1], perm [valid pairs], n_unrouted)."""
    ids = _c(topk_ids, np.int32)
    T, topk = ids.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm = np.empty(T * topk, np.int32)
    bad = _L().orc_moe_route(_p(ids), T, topk, E, _p(counts), _p(offsets), _p(perm))
    return counts, offsets, perm[: int(offsets[E])], int(bad)


def grouped_qgemm_moe(qx, dx, topk_ids, x_row_mode: int, qw4, dw):
    """y [T*topk, N] in (token, slot) order; rows of unrouted pairs are zero."""
    qx = _c(qx, np.int8)
    dx = _c(dx, np.float32)
    ids = _c(topk_ids, np.int32)
    qw4 = _c(qw4, np.uint8)
    dw = _c(dw, np.uint16)
    T, topk = ids.shape
    E, N = qw4.shape[0], qw4.shape[1]
    K = qx.shape[1]
    P = T * topk
    y = np.empty((P, N), np.float32)
    mag = np.empty((P, N), np.float64)
    bad = _L().orc_grouped_qgemm_moe(_p(qx), _p(dx), K, _p(ids), T, topk, x_row_mode,
                                     _p(qw4), _p(dw), E, N, _p(y), _p(mag))
    return y, mag, int(bad)


def silu_mul(gu: np.ndarray, F: int) -> np.ndarray:
    """h [P, F] binary64 = silu(gu[:, :F]) * gu[:, F:2F] (gu binary32 [P, >= 2F])."""
    gu = _c(gu, np.float32)
    P, ld = gu.shape
    h = np.empty((P, F), np.float64)
    _L().orc_silu_mul(_p(gu), P, F, ld, _p(h))
    return h


def moe_combine(y: np.ndarray, w: np.ndarray):
    """(out [T, N] binary64, mag [T, N]) = router-weighted sum of the topk rows of each token."""
    y = _c(y, np.float32)
    w = _c(w, np.float32)
    T, topk = w.shape
    N = y.shape[1]
    out = np.empty((T, N), np.float64)
    mag = np.empty((T, N), np.float64)
    _L().orc_moe_combine(_p(y), _p(w), T, topk, N, _p(out), _p(mag))
    return out, mag


def import_gguf(blocks: np.ndarray, N: int, K: int, wbits: int):
    """GGUF Q8_0 (wbits 8) / Q4_0 (wbits 4) blocks -> (codes [N, K] int8 or [N, K/2] uint8,
    scales [N, K/32] uint16)."""
    blocks = _c(blocks, np.uint8)
    q = np.empty((N, K if wbits == 8 else K // 2), np.int8 if wbits == 8 else np.uint8)
    d = np.empty((N, K // 32), np.uint16)
    _L().orc_import_gguf(_p(blocks), N, K, 1 if wbits == 4 else 0, _p(q), _p(d))
    return q, d


def splitk_merge(m: np.ndarray, l: np.ndarray, acc: np.ndarray):
    """(out [R, D], lse [R], mag [R, D]) in binary64 from split partials m, l [S, R], acc [S, R, D]."""
    m, l, acc = _c(m, np.float32), _c(l, np.float32), _c(acc, np.float32)
    S, R = m.shape
    D = acc.shape[2]
    out = np.empty((R, D), np.float64)
    lse = np.empty(R, np.float64)
    mag = np.empty((R, D), np.float64)
    _L().orc_splitk_merge(_p(m), _p(l), _p(acc), S, R, D, _p(out), _p(lse), _p(mag))
    return out, lse, mag


def kv3_codebook():
    """(levels [8], thresholds [7]) of the 3-bit Lloyd-Max quantizer of N(0, 1), binary64."""
    lv = np.empty(8, np.float64)
    th = np.empty(7, np.float64)
    _L().orc_kv3_codebook(_p(lv), _p(th))
    return lv, th


def wht(x: np.ndarray) -> np.ndarray:
    """Orthonormal Walsh-Hadamard transform (Sylvester order) of each row, binary64."""
    x = _c(x, np.float64)
    T, D = x.shape
    y = np.empty_like(x)
    _L().orc_wht(_p(x), T, D, _p(y))
    return y


def kv3_encode(x: np.ndarray):
    """x float32 [T, D] -> (codes uint32 [T, 3D/32], scales float32 [T], u binary64 [T, D])."""
    x = _c(x, np.float32)
    T, D = x.shape
    _, th = kv3_codebook()
    th32 = th.astype(np.float32)
    codes = np.empty((T, 3 * D // 32), np.uint32)
    scales = np.empty(T, np.float32)
    u = np.empty((T, D), np.float64)
    _L().orc_kv3_encode(_p(x), T, D, _p(th32), _p(codes), _p(scales), _p(u))
    return codes, scales, u


def kv3_decode(codes: np.ndarray, scales: np.ndarray, D: int) -> np.ndarray:
    """(codes uint32 [T, 3D/32], scales float32 [T]) -> x^ binary64 [T, D]."""
    codes = _c(codes, np.uint32)
    scales = _c(scales, np.float32)
    T = codes.shape[0]
    lv, _ = kv3_codebook()
    lv32 = lv.astype(np.float32)
    out = np.empty((T, D), np.float64)
    _L().orc_kv3_decode(_p(codes), _p(scales), T, D, _p(lv32), _p(out))
    return out

