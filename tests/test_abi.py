"""The C ABI library builds for sm_103a, loads, exports every entry point that
include/qgemm.h declares, and rejects bad arguments on the host before any
CUDA call (so these run without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qgemm.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\**(\w+)\s*\(", src, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    from block_quantized_integer_gb300 import _native
    return _native.load()


def test_header_parses():
    names = _declared()
    for must in ("quantize_act_q8", "qgemm_q8_0", "qgemm_q4_0", "grouped_qgemm_moe",
                 "moe_route", "qgemm_workspace_size", "qg_status_string"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    from block_quantized_integer_gb300 import _native
    for name in _declared():
        assert hasattr(lib, name), name
        assert name in _native.SIGNATURES, f"binding lacks {name}"


def test_wait_limit_entry_is_test_only_and_declared(lib):
    assert "qg_debug_set_wait_limit" in _declared()


def test_status_strings(lib):
    for code, name in enumerate(["QG_OK", "QG_ERR_INVALID_ARG", "QG_ERR_ALIGNMENT",
                                 "QG_ERR_WORKSPACE", "QG_ERR_CUDA", "QG_ERR_UNSUPPORTED"]):
        assert lib.qg_status_string(code).decode() == name


A = ctypes.c_void_p(0x10000)       # 16-byte aligned fake device addresses: never dereferenced
B = ctypes.c_void_p(0x20000)
C = ctypes.c_void_p(0x30000)
D = ctypes.c_void_p(0x40000)
Y = ctypes.c_void_p(0x50000)
NUL = ctypes.c_void_p(0)
S = ctypes.c_void_p(0)


def test_dense_validation(lib):
    f = lib.qgemm_q8_0
    assert f(A, B, 4, 256, 500, C, D, Y, 256, NUL, 0, S) == 1        # K % 32
    assert f(A, B, 4, 0, 512, C, D, Y, 256, NUL, 0, S) == 1          # N == 0
    assert f(A, B, -1, 256, 512, C, D, Y, 256, NUL, 0, S) == 1       # M < 0
    assert f(A, B, 4, 256, 512, C, D, Y, 255, NUL, 0, S) == 1        # ldy < N
    assert f(NUL, B, 4, 256, 512, C, D, Y, 256, NUL, 0, S) == 1      # null qx
    assert f(ctypes.c_void_p(0x10008), B, 4, 256, 512, C, D, Y, 256, NUL, 0, S) == 2
    assert f(A, B, 4, 256, 512, C, D, ctypes.c_void_p(0x50002), 256, NUL, 0, S) == 2
    assert f(A, B, 0, 256, 512, C, D, Y, 256, NUL, 0, S) == 0        # M == 0: no-op
    assert lib.qgemm_q8_0_ex(A, B, 9, 256, 512, C, D, Y, 256, NUL, 0, 1, S) == 5  # GEMV M>8
    assert lib.qgemm_q8_0_ex(A, B, 9, 256, 512, C, D, Y, 256, NUL, 0, 77, S) == 1


def test_fused_gemv_validation(lib):
    f = lib.qgemv_q8_0_f32
    assert f(A, 9, 512, 512, C, D, 256, Y, 256, S) == 1            # M > 8
    assert f(A, 4, 500, 500, C, D, 256, Y, 256, S) == 1            # K % 32
    assert f(A, 4, 512, 511, C, D, 256, Y, 256, S) == 1            # ldx < K
    assert f(A, 4, 512, 512, C, D, 256, Y, 255, S) == 1            # ldy < N
    assert f(NUL, 4, 512, 512, C, D, 256, Y, 256, S) == 1          # null x
    assert f(ctypes.c_void_p(0x10002), 4, 512, 512, C, D, 256, Y, 256, S) == 2
    assert f(A, 4, 512, 512, ctypes.c_void_p(0x30008), D, 256, Y, 256, S) == 2
    assert f(A, 0, 512, 512, C, D, 256, Y, 256, S) == 0            # M == 0: no-op
    # 8 rows x 24576: 221 KiB of codes and scales, above one block's share
    assert f(A, 8, 24576, 24576, C, D, 256, Y, 256, S) == 5


def test_quantize_validation(lib):
    assert lib.quantize_act_q8(A, 4, 48, 48, B, C, S) == 1            # K % 32
    assert lib.quantize_act_q8(A, 4, 64, 32, B, C, S) == 1            # ldx < K
    assert lib.quantize_act_q8(A, 0, 64, 64, B, C, S) == 0
    assert lib.quantize_act_q8(A, 4, 64, 64, ctypes.c_void_p(0x20001), C, S) == 2
    assert lib.quantize_weight_q8_0(A, 4, 40, B, C, S) == 1
    assert lib.quantize_weight_q4_0(NUL, 4, 64, B, C, S) == 1


def test_moe_validation_and_workspace(lib):
    ws = lib.qgemm_workspace_size(3, 0, 2048, 2048, 947, 8, 128)
    # counts E, offsets E+1, tile offsets E+1, perm T*topk (int32, 16-byte padded)
    assert ws >= 4 * (128 + 129 + 129 + 947 * 8)
    assert ws % 16 == 0
    assert lib.qgemm_workspace_size(1, 4, 256, 512, 0, 0, 0) == 0
    g = lib.grouped_qgemm_moe
    E = ctypes.c_void_p(0x60000)
    W = ctypes.c_void_p(0x70000)
    assert g(A, B, 947, 2048, C, 947, 8, 0, D, E, 128, 2048, Y, C, W, ws - 16, S) == 3
    assert g(A, B, 947, 2048, C, 947, 8, 0, D, E, 128, 2048, Y, C, NUL, ws, S) == 3
    assert g(A, B, 946, 2048, C, 947, 8, 0, D, E, 128, 2048, Y, C, W, ws, S) == 1  # rows_x < T
    assert g(A, B, 947, 2048, C, 947, 8, 1, D, E, 128, 2048, Y, C, W, ws, S) == 1  # mode 1 rows
    assert g(A, B, 947, 2048, C, 947, 8, 2, D, E, 128, 2048, Y, C, W, ws, S) == 1
    assert g(A, B, 947, 2048, C, 947, 8, 0, D, E, 2000, 2048, Y, C, W, ws, S) == 1  # E > 1024
    assert lib.moe_route(A, 10, 2, 2000, B, C, D, Y, S) == 1
    assert lib.moe_route(NUL, 10, 2, 16, B, C, D, Y, S) == 1     # null ids with T > 0
    assert g(A, B, 0, 2048, C, 0, 8, 0, D, E, 128, 2048, Y, C, W, ws, S) == 0   # T == 0: no-op
    # T * topk past int64 range: rejected before the product is formed
    huge = (1 << 62) + 1
    assert g(A, B, huge, 2048, C, huge, 8, 0, D, E, 128, 2048, Y, C, W, ws, S) == 1
    assert lib.moe_route(A, huge, 8, 16, B, C, D, Y, S) == 1
    assert lib.qgemm_workspace_size(3, 0, 2048, 2048, huge, 8, 128) == 0
    assert lib.grouped_qgemm_moe_noalloc(A, B, huge, 2048, C, huge, 8, 0, D, E, 128, 2048, Y, C,
                                         S) == 5
    assert lib.grouped_qgemm_moe_noalloc(A, B, 70000, 2048, C, 70000, 1, 0, D, E, 128, 2048, Y,
                                         C, S) == 5      # more routed pairs than the array holds
    assert lib.grouped_qgemm_moe_noalloc(A, B, 947, 2048, C, 947, 8, 0, D, E, 1025, 2048, Y,
                                         C, S) == 5      # more experts than the array holds


def test_dense_tc_workspace_size(lib):
    """The tensor-core product's workspace as documented: binary16 activation codes, the
    transposed binary32 weight scales, binary16 weight codes, each padded to 16 bytes, plus
    whole 64 KiB partial tiles for a tail split (none without a device: 0 SMs)."""
    def a16(v):
        return (v + 15) // 16 * 16
    for op in (1, 2):                                   # Q8_0, Q4_0
        for M, N, K in ((300, 130, 768), (9, 1, 256), (2048, 12288, 4096), (4000, 33, 512)):
            G = K // 32
            base = a16(M * K * 2) + a16(G * ((N + 31) // 32 * 32) * 4) + a16(N * K * 2)
            ws = lib.qgemm_workspace_size(op, M, N, K, 0, 0, 0)
            assert ws >= base and (ws - base) % 65536 == 0 and ws - base <= 1024 * 65536
    assert lib.qgemm_workspace_size(1, 300, 130, 96, 0, 0, 0) == 0     # K % 256 != 0: no TMA path


def test_debug_group_dots_validation(lib):
    f = lib.qgemm_debug_group_dots
    ws = lib.qgemm_workspace_size(4, 16, 64, 512, 0, 0, 0)
    # dx [16][16] f32 + dw [64][16] f16 + y [16][64] f32 + the tcgen05 workspace for M = 9..16
    assert ws >= 16 * 16 * 4 + 64 * 16 * 2 + 16 * 64 * 4 and ws % 16 == 0
    W = ctypes.c_void_p(0x70000)
    assert f(A, 16, 64, 500, C, 8, 0, Y, W, ws, S) == 1       # K % 32
    assert f(A, 16, 64, 512, C, 5, 0, Y, W, ws, S) == 1       # bits
    assert f(A, 16, 64, 512, C, 8, 0, NUL, W, ws, S) == 1     # null S
    assert f(ctypes.c_void_p(0x10008), 16, 64, 512, C, 8, 0, Y, W, ws, S) == 2
    assert f(A, 16, 64, 512, C, 8, 0, Y, W, ws - 16, S) == 3  # workspace too small
    assert f(A, 16, 64, 512, C, 8, 0, Y, NUL, ws, S) == 3
    assert f(A, 0, 64, 512, C, 8, 0, Y, W, ws, S) == 0        # M == 0: no-op


def test_moe_ffn_steps_validation(lib):
    f = lib.moe_swiglu_quant
    assert f(A, 4, 48, 96, B, C, S) == 1            # F % 32
    assert f(A, 4, 64, 100, B, C, S) == 1           # ldgu < 2F
    assert f(A, -1, 64, 128, B, C, S) == 1
    assert f(A, 0, 64, 128, B, C, S) == 0           # P == 0: no-op
    assert f(NUL, 4, 64, 128, B, C, S) == 1
    assert f(A, 4, 64, 128, ctypes.c_void_p(0x20004), C, S) == 2   # qh not 16-byte aligned
    g = lib.moe_combine
    assert g(A, B, 4, 0, 64, C, S) == 1             # topk
    assert g(A, B, 4, 8, 0, C, S) == 1              # N
    assert g(A, B, 0, 8, 64, C, S) == 0             # T == 0: no-op
    assert g(A, NUL, 4, 8, 64, C, S) == 1
    assert g(A, B, 4, 8, 64, ctypes.c_void_p(0x30002), S) == 2


def test_gguf_import_validation(lib):
    f = lib.import_gguf_q8_0
    assert f(A, 4, 48, B, C, S) == 1                 # K % 32
    assert f(A, -1, 64, B, C, S) == 1
    assert f(A, 0, 64, B, C, S) == 0                 # N == 0: no-op
    assert f(NUL, 4, 64, B, C, S) == 1
    assert f(ctypes.c_void_p(0x10001), 4, 64, B, C, S) == 2     # blocks 2-byte aligned
    assert lib.import_gguf_q4_0(A, 4, 64, ctypes.c_void_p(0x20008), C, S) == 2


def test_splitk_merge_validation(lib):
    f = lib.attn_splitk_merge
    assert f(A, B, C, 0, 4, 128, D, NUL, S) == 1          # S >= 1
    assert f(A, B, C, 65, 4, 128, D, NUL, S) == 1         # S <= 64
    assert f(A, B, C, 4, 4, 0, D, NUL, S) == 1            # D >= 1
    assert f(A, B, C, 4, 0, 128, D, NUL, S) == 0          # R == 0: no-op
    assert f(A, NUL, C, 4, 4, 128, D, NUL, S) == 1
    assert f(A, B, C, 4, 4, 128, ctypes.c_void_p(0x40002), NUL, S) == 2


def test_kv3_library_codebook_matches_oracle(lib):
    """The library computes its codebook on the host; it equals the oracle's, rounded."""
    import numpy as np
    import oracle
    lv = np.zeros(8, np.float32)
    th = np.zeros(7, np.float32)
    lib.qg_kv3_codebook(lv.ctypes.data_as(ctypes.c_void_p), th.ctypes.data_as(ctypes.c_void_p))
    olv, oth = oracle.kv3_codebook()
    assert np.array_equal(lv, olv.astype(np.float32))
    assert np.array_equal(th, oth.astype(np.float32))


def test_kv3_validation(lib):
    assert lib.kv3_encode(A, 4, 96, 96, B, C, S) == 1        # D not 64/128/256
    assert lib.kv3_encode(A, 4, 128, 100, B, C, S) == 1      # ldx < D
    assert lib.kv3_encode(A, 0, 128, 128, B, C, S) == 0      # T == 0: no-op
    assert lib.kv3_encode(NUL, 4, 128, 128, B, C, S) == 1
    assert lib.kv3_decode(A, ctypes.c_void_p(0x20002), 4, 128, C, 128, S) == 2
