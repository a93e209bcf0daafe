"""Block-quantized integer GEMM/GEMV (Q8_0 / Q4_0 weights, int8 activations)
for NVIDIA GB300 (sm_103a).

Thin binding over the C ABI in ``include/qgemm.h`` (``libqgemm.so``): the
functions below only check tensor dtypes/devices, allocate outputs with
PyTorch when the caller passes none, and forward pointers, sizes and the
current CUDA stream.  Every step of the computation runs in the library's CUDA
kernels; nothing here falls back to the CPU.

Tensor conventions (row-major, K contiguous, G = K // 32):
  x   float32 [M, K]         qx int8 [M, K]      dx float32 [M, G]
  qw  int8    [N, K]         qw4 uint8 [N, K/2]  dw float16 [N, G] (the binary16
                                                    scales, passed as bit patterns)
  y   float32 [M, N]
"""
from __future__ import annotations

import ctypes

import torch

from . import _native
from ._native import QGError

__all__ = [
    "QGError", "ALGO_AUTO", "ALGO_GEMV", "ALGO_MMA", "ALGO_TCGEN05",
    "quantize_act_q8", "quantize_weight_q8_0", "quantize_weight_q4_0",
    "qgemm_q8_0", "qgemm_q4_0", "qgemv_q8_0_f32", "moe_route", "grouped_qgemm_moe", "grouped_qgemm_moe_noalloc",
    "import_gguf_q8_0", "import_gguf_q4_0",
    "attn_splitk_merge", "kv3_encode", "kv3_decode", "kv3_codebook",
    "moe_swiglu_quant", "moe_combine",
    "workspace_size", "debug_group_dots",
    "sm_count", "device_error", "debug_set_wait_limit",
]

ALGO_AUTO, ALGO_GEMV, ALGO_MMA, ALGO_TCGEN05 = 0, 1, 2, 3
OP_QGEMM_Q8_0, OP_QGEMM_Q4_0, OP_GROUPED_MOE, OP_DEBUG_GROUP_DOTS = 1, 2, 3, 4


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(dev):
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _need(t, dtype, name, dev=None, rows_strided=False):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dev is not None and t.device != dev:
        raise ValueError(f"{name} is on {t.device}, expected {dev}")
    if rows_strided:
        if t.dim() != 2 or t.stride(1) != 1:
            raise ValueError(f"{name} must be 2-D with unit column stride")
    elif not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def sm_count() -> int:
    return int(_native.load().qg_device_sm_count())


def device_error() -> int:
    """Read and clear the tensor-core kernels' device error word (0 = none)."""
    return int(_native.load().qg_device_error())


def debug_set_wait_limit(cycles: int) -> None:
    """Test-only: SM cycles a tensor-core pipeline wait may last before the kernel
    gives up and sets the device error word (cycles <= 0: the default, ~2 s)."""
    _native.call("qg_debug_set_wait_limit", int(cycles))


def workspace_size(op: int, M=0, N=0, K=0, T=0, topk=0, E=0) -> int:
    return int(_native.load().qgemm_workspace_size(op, M, N, K, T, topk, E))


def quantize_act_q8(x: torch.Tensor, qx: torch.Tensor | None = None,
                    dx: torch.Tensor | None = None):
    """x float32 [M, K] -> (qx int8 [M, K], dx float32 [M, K/32])."""
    _need(x, torch.float32, "x", rows_strided=True)
    M, K = x.shape
    if qx is None:
        qx = torch.empty((M, K), dtype=torch.int8, device=x.device)
    if dx is None:
        dx = torch.empty((M, K // 32), dtype=torch.float32, device=x.device)
    _need(qx, torch.int8, "qx", x.device)
    _need(dx, torch.float32, "dx", x.device)
    if tuple(qx.shape) != (M, K) or tuple(dx.shape) != (M, K // 32):
        raise ValueError(f"qx must be [{M}, {K}] and dx [{M}, {K // 32}]")
    _native.call("quantize_act_q8", _ptr(x), M, K, x.stride(0), _ptr(qx), _ptr(dx),
                 _stream(x.device))
    return qx, dx


def quantize_weight_q8_0(w: torch.Tensor):
    """w float32 [N, K] -> (qw int8 [N, K], dw float16 [N, K/32])."""
    _need(w, torch.float32, "w")
    N, K = w.shape
    qw = torch.empty((N, K), dtype=torch.int8, device=w.device)
    dw = torch.empty((N, K // 32), dtype=torch.float16, device=w.device)
    _native.call("quantize_weight_q8_0", _ptr(w), N, K, _ptr(qw), _ptr(dw), _stream(w.device))
    return qw, dw


def quantize_weight_q4_0(w: torch.Tensor):
    """w float32 [N, K] -> (qw4 uint8 [N, K/2], dw float16 [N, K/32])."""
    _need(w, torch.float32, "w")
    N, K = w.shape
    qw4 = torch.empty((N, K // 2), dtype=torch.uint8, device=w.device)
    dw = torch.empty((N, K // 32), dtype=torch.float16, device=w.device)
    _native.call("quantize_weight_q4_0", _ptr(w), N, K, _ptr(qw4), _ptr(dw), _stream(w.device))
    return qw4, dw


def _dense(name, qx, dx, qw, dw, y, algo, workspace, wdtype, kfac):
    # shapes first (they need no device), then dtypes and devices
    for t, nm in ((qx, "qx"), (dx, "dx"), (qw, "qw"), (dw, "dw")):
        if not isinstance(t, torch.Tensor) or t.dim() != 2:
            raise ValueError(f"{nm} must be a 2-D tensor")
    M, K = qx.shape
    N = qw.shape[0]
    if qw.shape[1] * kfac != K or dw.shape != (N, K // 32) or dx.shape != (M, K // 32):
        raise ValueError("shape mismatch between qx/dx/qw/dw")
    if y is not None:
        if not isinstance(y, torch.Tensor) or y.dim() != 2 or y.stride(1) != 1:
            raise ValueError("y must be a 2-D tensor with unit column stride")
        if y.shape[0] < M or y.shape[1] < N:
            raise ValueError(f"y must have at least [{M}, {N}] elements, got {tuple(y.shape)}")
    _need(qx, torch.int8, "qx")
    dev = qx.device
    _need(dx, torch.float32, "dx", dev)
    _need(qw, wdtype, "qw", dev)
    _need(dw, torch.float16, "dw", dev)
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
    elif y.dtype != torch.float32 or y.device != dev:
        raise ValueError("y must be float32 on the same device")
    if workspace is None:
        op = OP_QGEMM_Q8_0 if kfac == 1 else OP_QGEMM_Q4_0
        nbytes = workspace_size(op, M, N, K)
        if algo == ALGO_TCGEN05:      # explicit tensor-core path at any M
            nbytes = max(nbytes, workspace_size(op, max(M, 9), N, K))
        if nbytes:
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    ws_ptr, ws_bytes = ctypes.c_void_p(0), 0
    if workspace is not None:
        ws_ptr, ws_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    _native.call(name, _ptr(qx), _ptr(dx), M, N, K, _ptr(qw), _ptr(dw), _ptr(y), y.stride(0),
                 ws_ptr, ws_bytes, int(algo), _stream(dev))
    return y


def qgemv_q8_0_f32(x, qw, dw, y=None):
    """Decode product from binary32 activations x [M, K] (M <= 8, rows may be
    strided): the activation quantization runs inside the GEMV; y equals
    qgemm_q8_0(*quantize_act_q8(x), qw, dw) bit for bit."""
    _need(x, torch.float32, "x", rows_strided=True)
    dev = x.device
    _need(qw, torch.int8, "qw", dev)
    _need(dw, torch.float16, "dw", dev)
    M, K = x.shape
    N = qw.shape[0]
    if qw.shape[1] != K or dw.shape != (N, K // 32):
        raise ValueError("shape mismatch between x/qw/dw")
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
    elif y.dtype != torch.float32 or y.device != dev or y.stride(1) != 1 or tuple(y.shape) != (M, N):
        raise ValueError("y must be float32 [M, N] on the same device with unit column stride")
    _native.call("qgemv_q8_0_f32", _ptr(x), M, K, x.stride(0), _ptr(qw), _ptr(dw), N, _ptr(y),
                 y.stride(0), _stream(dev))
    return y


def qgemm_q8_0(qx, dx, qw, dw, y=None, algo: int = ALGO_AUTO, workspace=None):
    """y[m,n] = sum_g dw[n,g] dx[m,g] sum_{k in g} qx[m,k] qw[n,k] (Q8_0 weights)."""
    return _dense("qgemm_q8_0_ex", qx, dx, qw, dw, y, algo, workspace, torch.int8, 1)


def qgemm_q4_0(qx, dx, qw4, dw, y=None, algo: int = ALGO_AUTO, workspace=None):
    """As qgemm_q8_0 with Q4_0 weights qw4 uint8 [N, K/2]."""
    return _dense("qgemm_q4_0_ex", qx, dx, qw4, dw, y, algo, workspace, torch.uint8, 2)


def _import_gguf(name, blocks, N, K, bytes_per_block, code_dtype, code_cols):
    _need(blocks, torch.uint8, "blocks")
    if blocks.numel() != N * (K // 32) * bytes_per_block:
        raise ValueError(f"blocks must hold N * K/32 blocks of {bytes_per_block} bytes")
    dev = blocks.device
    q = torch.empty((N, code_cols), dtype=code_dtype, device=dev)
    dw = torch.empty((N, K // 32), dtype=torch.float16, device=dev)
    _native.call(name, _ptr(blocks), N, K, _ptr(q), _ptr(dw), _stream(dev))
    return q, dw


def import_gguf_q8_0(blocks: torch.Tensor, N: int, K: int):
    """GGUF Q8_0 blocks (uint8, N * K/32 * 34 bytes) -> (qw int8 [N, K], dw float16 [N, K/32])."""
    return _import_gguf("import_gguf_q8_0", blocks, N, K, 34, torch.int8, K)


def import_gguf_q4_0(blocks: torch.Tensor, N: int, K: int):
    """GGUF Q4_0 blocks (uint8, N * K/32 * 18 bytes) -> (qw4 uint8 [N, K/2], dw float16 [N, K/32])."""
    return _import_gguf("import_gguf_q4_0", blocks, N, K, 18, torch.uint8, K // 2)


def kv3_encode(x: torch.Tensor):
    """x float32 [T, D] (D = 64, 128, 256) -> (codes int32 [T, 3D/32] holding the bit-plane
    words, scales float32 [T])."""
    _need(x, torch.float32, "x", rows_strided=True)
    T, D = x.shape
    codes = torch.empty((T, 3 * D // 32), dtype=torch.int32, device=x.device)
    scales = torch.empty(T, dtype=torch.float32, device=x.device)
    _native.call("kv3_encode", _ptr(x), T, D, x.stride(0), _ptr(codes), _ptr(scales),
                 _stream(x.device))
    return codes, scales


def kv3_decode(codes: torch.Tensor, scales: torch.Tensor, D: int, out: torch.Tensor = None):
    """(codes int32 [T, 3D/32], scales float32 [T]) -> x^ float32 [T, D] (written into
    `out`, rows may be strided, when given)."""
    _need(codes, torch.int32, "codes")
    _need(scales, torch.float32, "scales", codes.device)
    T = codes.shape[0]
    if out is None:
        out = torch.empty((T, D), dtype=torch.float32, device=codes.device)
    else:
        _need(out, torch.float32, "out", codes.device, rows_strided=True)
        if tuple(out.shape) != (T, D):
            raise ValueError(f"out must be [{T}, {D}], got {tuple(out.shape)}")
    _native.call("kv3_decode", _ptr(codes), _ptr(scales), T, D, _ptr(out), out.stride(0),
                 _stream(codes.device))
    return out


def kv3_codebook():
    """(levels [8], thresholds [7]) float32 numpy arrays of the codec in use."""
    import numpy as np
    lv = np.zeros(8, np.float32)
    th = np.zeros(7, np.float32)
    _native.load().qg_kv3_codebook(lv.ctypes.data_as(ctypes.c_void_p), th.ctypes.data_as(ctypes.c_void_p))
    return lv, th


def attn_splitk_merge(m: torch.Tensor, l: torch.Tensor, acc: torch.Tensor, want_lse: bool = True):
    """Split-K attention partials m, l float32 [S, R], acc float32 [S, R, D] ->
    (out float32 [R, D], lse float32 [R] or None), splits merged in index order."""
    _need(m, torch.float32, "m")
    dev = m.device
    _need(l, torch.float32, "l", dev)
    _need(acc, torch.float32, "acc", dev)
    S, R = m.shape
    D = acc.shape[2]
    if l.shape != (S, R) or acc.shape[:2] != (S, R):
        raise ValueError("shape mismatch between m/l/acc")
    out = torch.empty((R, D), dtype=torch.float32, device=dev)
    lse = torch.empty(R, dtype=torch.float32, device=dev) if want_lse else None
    _native.call("attn_splitk_merge", _ptr(m), _ptr(l), _ptr(acc), S, R, D, _ptr(out), _ptr(lse),
                 _stream(dev))
    return out, lse


def moe_swiglu_quant(gu: torch.Tensor, F: int | None = None):
    """gu float32 [P, >= 2F] (gate columns [0, F), up [F, 2F)) ->
    (qh int8 [P, F], dh float32 [P, F/32]): h = silu(gate) * up quantized per 32-group."""
    _need(gu, torch.float32, "gu", rows_strided=True)
    P = gu.shape[0]
    if F is None:
        F = gu.shape[1] // 2
    if gu.shape[1] < 2 * F:
        raise ValueError(f"gu must have at least 2F = {2 * F} columns, got {gu.shape[1]}")
    qh = torch.empty((P, F), dtype=torch.int8, device=gu.device)
    dh = torch.empty((P, F // 32), dtype=torch.float32, device=gu.device)
    _native.call("moe_swiglu_quant", _ptr(gu), P, F, gu.stride(0), _ptr(qh), _ptr(dh),
                 _stream(gu.device))
    return qh, dh


def moe_combine(y: torch.Tensor, w: torch.Tensor, out: torch.Tensor | None = None):
    """y float32 [T*topk, N] (token, slot order), w float32 [T, topk] -> out [T, N] =
    sum over slots of w * y, slot order."""
    _need(y, torch.float32, "y")
    dev = y.device
    _need(w, torch.float32, "w", dev)
    T, topk = w.shape
    N = y.shape[1]
    if y.shape[0] != T * topk:
        raise ValueError("y must have T * topk rows")
    if out is None:
        out = torch.empty((T, N), dtype=torch.float32, device=dev)
    else:
        _need(out, torch.float32, "out", dev)
        if tuple(out.shape) != (T, N):
            raise ValueError(f"out must be [{T}, {N}], got {tuple(out.shape)}")
    _native.call("moe_combine", _ptr(y), _ptr(w), T, topk, N, _ptr(out), _stream(dev))
    return out


def debug_group_dots(qx, qw, bits: int, algo: int = ALGO_AUTO):
    """Test-only: the exact group dots S int32 [M, N, K/32] as the product kernel
    `algo` forms them (qw int8 [N, K] for bits 8, uint8 [N, K/2] for bits 4)."""
    _need(qx, torch.int8, "qx")
    dev = qx.device
    _need(qw, torch.int8 if bits == 8 else torch.uint8, "qw", dev)
    M, K = qx.shape
    N = qw.shape[0]
    if qw.shape[1] * (1 if bits == 8 else 2) != K:
        raise ValueError("shape mismatch between qx and qw")
    S = torch.empty((M, N, K // 32), dtype=torch.int32, device=dev)
    nbytes = workspace_size(OP_DEBUG_GROUP_DOTS, M, N, K)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)
    _native.call("qgemm_debug_group_dots", _ptr(qx), M, N, K, _ptr(qw), int(bits), int(algo),
                 _ptr(S), _ptr(ws), ws.numel(), _stream(dev))
    return S


def moe_route(topk_ids: torch.Tensor, E: int, d_err: torch.Tensor | None = None):
    """topk_ids int32 [T, topk] -> (counts [E], offsets [E+1], perm [T*topk], d_err [1])."""
    _need(topk_ids, torch.int32, "topk_ids")
    dev = topk_ids.device
    T, topk = topk_ids.shape
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(max(T * topk, 1), dtype=torch.int32, device=dev)
    if d_err is None:
        d_err = torch.zeros(1, dtype=torch.int32, device=dev)
    _native.call("moe_route", _ptr(topk_ids), T, topk, E, _ptr(counts), _ptr(offsets),
                 _ptr(perm), _ptr(d_err), _stream(dev))
    return counts, offsets, perm, d_err


def _moe_shapes(qx, dx, topk_ids, qw4, dw, y, d_err):
    """Shape checks of the grouped MoE product, before anything reaches the
    library: a short y or weight plane would otherwise be written or read past
    its end by the kernels.  Returns (rows_x, K, T, topk, E, N)."""
    for t, nm, nd in ((qx, "qx", 2), (dx, "dx", 2), (topk_ids, "topk_ids", 2), (qw4, "qw4", 3),
                      (dw, "dw", 3)):
        if not isinstance(t, torch.Tensor) or t.dim() != nd:
            raise ValueError(f"{nm} must be a {nd}-D tensor")
    rows_x, K = qx.shape
    T, topk = topk_ids.shape
    E, N = qw4.shape[0], qw4.shape[1]
    if K % 32 != 0:
        raise ValueError(f"K = {K} is not a multiple of 32")
    if tuple(dx.shape) != (rows_x, K // 32):
        raise ValueError(f"dx must be [{rows_x}, {K // 32}], got {tuple(dx.shape)}")
    if tuple(qw4.shape) != (E, N, K // 2):
        raise ValueError(f"qw4 must be [E, N, {K // 2}], got {tuple(qw4.shape)}")
    if tuple(dw.shape) != (E, N, K // 32):
        raise ValueError(f"dw must be [{E}, {N}, {K // 32}], got {tuple(dw.shape)}")
    if y is not None and (not isinstance(y, torch.Tensor) or tuple(y.shape) != (T * topk, N)
                          or not y.is_contiguous()):
        raise ValueError(f"y must be a contiguous [{T * topk}, {N}] tensor")
    if d_err is not None and (not isinstance(d_err, torch.Tensor) or d_err.numel() < 1):
        raise ValueError("d_err must hold at least one int32")
    return rows_x, K, T, topk, E, N


def grouped_qgemm_moe(qx, dx, topk_ids, x_row_mode: int, qw4, dw, y=None, d_err=None,
                      workspace=None):
    """Per routed pair p: y[p] = x_row(p) @ W_{e(p)}^T with Q4_0 expert weights
    qw4 [E, N, K/2], dw float16 [E, N, K/32]; y [T*topk, N] in (token, slot) order."""
    rows_x, K, T, topk, E, N = _moe_shapes(qx, dx, topk_ids, qw4, dw, y, d_err)
    _need(qx, torch.int8, "qx")
    dev = qx.device
    _need(dx, torch.float32, "dx", dev)
    _need(topk_ids, torch.int32, "topk_ids", dev)
    _need(qw4, torch.uint8, "qw4", dev)
    _need(dw, torch.float16, "dw", dev)
    if y is None:
        y = torch.empty((T * topk, N), dtype=torch.float32, device=dev)
    else:
        _need(y, torch.float32, "y", dev)
    if d_err is None:
        d_err = torch.zeros(1, dtype=torch.int32, device=dev)
    else:
        _need(d_err, torch.int32, "d_err", dev)
    if workspace is not None:
        _need(workspace, torch.uint8, "workspace", dev)
    if workspace is None:
        nbytes = workspace_size(OP_GROUPED_MOE, 0, N, K, T, topk, E)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)
    _native.call("grouped_qgemm_moe", _ptr(qx), _ptr(dx), rows_x, K, _ptr(topk_ids), T, topk,
                 int(x_row_mode), _ptr(qw4), _ptr(dw), E, N, _ptr(y), _ptr(d_err),
                 _ptr(workspace), workspace.numel(), _stream(dev))
    return y, d_err


def grouped_qgemm_moe_noalloc(qx, dx, topk_ids, x_row_mode: int, qw4, dw, y, d_err):
    """grouped_qgemm_moe through the entry point that allocates nothing: the
    routing scratch is a fixed array inside the library (at most 65536 routed
    pairs and 1024 experts).  For callers that cannot allocate device memory,
    y and d_err (zeroed by the caller) must be passed in."""
    if y is None or d_err is None:
        raise ValueError("y and d_err must be passed in: this entry point allocates nothing")
    rows_x, K, T, topk, E, N = _moe_shapes(qx, dx, topk_ids, qw4, dw, y, d_err)
    _need(qx, torch.int8, "qx")
    dev = qx.device
    _need(dx, torch.float32, "dx", dev)
    _need(topk_ids, torch.int32, "topk_ids", dev)
    _need(qw4, torch.uint8, "qw4", dev)
    _need(dw, torch.float16, "dw", dev)
    _need(y, torch.float32, "y", dev)
    _need(d_err, torch.int32, "d_err", dev)
    _native.call("grouped_qgemm_moe_noalloc", _ptr(qx), _ptr(dx), rows_x, K, _ptr(topk_ids), T,
                 topk, int(x_row_mode), _ptr(qw4), _ptr(dw), E, N, _ptr(y), _ptr(d_err),
                 _stream(dev))
    return y, d_err
