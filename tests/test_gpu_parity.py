"""GPU parity: the CUDA kernels behind the C ABI against the CPU oracle.

Bar: bit-exact for the quantized codes, the scales and every group's integer
dot product S; y within |y - y_ref| <= 1e-5 * sum_g |dw dx S_g| per element
(binary32 output, reordered sums).  Small cases compare every output; the
full-size workloads (in the launch configuration the benchmark uses) compare
sampled rows the oracle computes one by one.
"""
import numpy as np
import pytest
import torch

import oracle
import block_quantized_integer_gb300 as qg
from block_quantized_integer_gb300 import inputs
from helpers import assert_close, dev, to_dev, to_np

pytestmark = pytest.mark.gpu

DENSE_ALGOS = [qg.ALGO_GEMV, qg.ALGO_MMA, qg.ALGO_TCGEN05]


def _sync():
    torch.cuda.synchronize()


# ------------------------------------------------------------------ quantizers

@pytest.mark.parametrize("M,K,ldx", [(4, 512, 512), (1, 4096, 4096), (37, 96, 96), (3, 32, 32),
                                     (5, 160, 200), (2, 64, 67)])
def test_quantize_act_bit_exact(M, K, ldx):
    rng = np.random.default_rng(M * 1000 + K)
    xf = rng.standard_normal((M, ldx)).astype(np.float32)
    xf[:, rng.choice(ldx, max(1, ldx // 50), replace=False)] *= 25
    xf[0, :32] = 0.0
    if M > 1:
        xf[1, :32] *= np.float32(1e-39)          # subnormal inputs and scales
    x = xf[:, :K]
    qx_ref, dx_ref = oracle.quantize_act_q8(x)
    xt = to_dev(xf)[:, :K]                       # row stride ldx
    qx, dx = qg.quantize_act_q8(xt)
    _sync()
    assert np.array_equal(to_np(qx), qx_ref)
    assert np.array_equal(to_np(dx).view(np.uint32), dx_ref.view(np.uint32))


def test_quantize_act_golden_ties():
    rows = []
    import os
    for line in open(os.path.join(os.path.dirname(__file__), "golden", "q8_act_ties.txt")):
        if line.strip() and not line.startswith("#") and not line.startswith("d "):
            rows.append(line.split())
    x = np.array([[float(r[0]) for r in rows]], np.float32)
    qx, dx = qg.quantize_act_q8(to_dev(x))
    _sync()
    assert to_np(qx)[0].tolist() == [int(r[1]) for r in rows]
    assert to_np(dx)[0, 0] == 1.0


def test_quantize_act_near_ties():
    """Quotients x / d placed within 1e-6 .. 5e-4 of a half-integer, and on it, where
    any shortcut past the binary32 division would show first: codes bit-exact with
    the oracle's, also through the GEMV that quantizes its own activations."""
    rng = np.random.default_rng(4242)
    M, K = 128, 1024
    G = M * K // 32
    amax = rng.uniform(0.5, 3.0, G).astype(np.float32)
    d = amax / np.float32(127.0)                       # binary32 quotients, as the rule
    k = rng.integers(-126, 126, (G, 31)).astype(np.float64)
    off = rng.choice([-5e-4, -3e-4, -2e-4, -3e-5, -1e-5, -1e-6, 0.0, 1e-6, 1e-5, 3e-5, 2e-4,
                      3e-4, 5e-4], (G, 31))
    g = np.empty((G, 32), np.float32)
    g[:, 0] = amax
    g[:, 1:] = ((k + 0.5 + off) * d[:, None].astype(np.float64)).astype(np.float32)
    x = g.reshape(M, K)
    qx_ref, dx_ref = oracle.quantize_act_q8(x)
    qx, dx = qg.quantize_act_q8(to_dev(x))
    _sync()
    assert np.array_equal(to_np(qx), qx_ref)
    assert np.array_equal(to_np(dx).view(np.uint32), dx_ref.view(np.uint32))
    w = (rng.standard_normal((64, K)) * 0.02).astype(np.float32)
    qw, dw = qg.quantize_weight_q8_0(to_dev(w))
    for m0 in range(0, M, 8):                          # the fused GEMV, 8 rows at a time
        xs = to_dev(x[m0:m0 + 8])
        y_fused = qg.qgemv_q8_0_f32(xs, qw, dw)
        y_two = qg.qgemm_q8_0(qx[m0:m0 + 8].contiguous(), dx[m0:m0 + 8].contiguous(), qw, dw)
        _sync()
        assert torch.equal(y_fused, y_two)


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("N,K", [(256, 512), (300, 96), (7, 32), (1024, 2048)])
def test_quantize_weight_bit_exact(bits, N, K):
    rng = np.random.default_rng(N + K + bits)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    w[0, :32] = 0.0
    w[min(1, N - 1), 32 % K:32 % K + 32] *= np.float32(1e-4)   # subnormal binary16 scales
    if bits == 8:
        q_ref, d_ref = oracle.quantize_w_q8_0(w)
        q, d = qg.quantize_weight_q8_0(to_dev(w))
    else:
        q_ref, d_ref = oracle.quantize_w_q4_0(w)
        q, d = qg.quantize_weight_q4_0(to_dev(w))
    _sync()
    assert np.array_equal(to_np(q), q_ref)
    assert np.array_equal(to_np(d), d_ref)


# ------------------------------------------------------------------ group dots

def _gemm(bits, algo, qx, dx, qw, dw, y=None):
    f = qg.qgemm_q8_0 if bits == 8 else qg.qgemm_q4_0
    return f(qx, dx, qw, dw, y=y, algo=algo)


@pytest.mark.parametrize("algo", DENSE_ALGOS)
@pytest.mark.parametrize("bits", [8, 4])
def test_group_dots_exact(algo, bits):
    """With dx = 1 and dw = 1 on group g and 0 elsewhere, y = S[:, :, g] exactly."""
    M = 5 if algo == qg.ALGO_GEMV else 70
    N, K = (150, 256) if algo != qg.ALGO_TCGEN05 else (300, 512)
    G = K // 32
    rng = np.random.default_rng(17 + bits + algo)
    qx = rng.integers(-127, 128, (M, K)).astype(np.int8)
    qx[0, :32] = 127
    if bits == 8:
        qw = rng.integers(-127, 128, (N, K)).astype(np.int8)
        qw[0, :32] = 127
        qw[1, :32] = -127
    else:
        qw = rng.integers(0, 256, (N, K // 2)).astype(np.uint8)
    S = oracle.group_dots(qx, qw, K, bits)
    dx = np.ones((M, G), np.float32)
    qx_t, dx_t, qw_t = to_dev(qx), to_dev(dx), to_dev(qw)
    for g in range(G):
        dw = np.zeros((N, G), np.float16)
        dw[:, g] = 1.0
        y = _gemm(bits, algo, qx_t, dx_t, qw_t, to_dev(dw.view(np.uint16)))
        _sync()
        assert np.array_equal(to_np(y), S[:, :, g].astype(np.float32)), f"group {g}"
    if bits == 8:
        assert S[0, 0, 0] == 32 * 127 * 127 and S[0, 1, 0] == -32 * 127 * 127
    assert qg.device_error() == 0


@pytest.mark.parametrize("algo,M,N,K", [(qg.ALGO_GEMV, 3, 70, 96), (qg.ALGO_GEMV, 8, 33, 512),
                                         (qg.ALGO_MMA, 37, 150, 256), (qg.ALGO_TCGEN05, 130, 200, 512),
                                         (qg.ALGO_AUTO, 9, 129, 256)])
@pytest.mark.parametrize("bits", [8, 4])
def test_debug_group_dots_bit_exact(algo, M, N, K, bits):
    """The C-ABI group-dot readout of each kernel equals the oracle's int64 dots."""
    rng = np.random.default_rng(1000 + 7 * M + bits + algo)
    qx = rng.integers(-127, 128, (M, K)).astype(np.int8)
    qx[0, :32] = 127
    qx[-1, -32:] = -127
    if bits == 8:
        qw = rng.integers(-127, 128, (N, K)).astype(np.int8)
        qw[0, :32] = 127
        qw[-1, -32:] = 127
    else:
        qw = rng.integers(0, 256, (N, K // 2)).astype(np.uint8)
        qw[0, :16] = 0x00                  # all elements -8
    S = qg.debug_group_dots(to_dev(qx), to_dev(qw), bits, algo)
    _sync()
    ref = oracle.group_dots(qx, qw, K, bits)
    assert np.array_equal(to_np(S).astype(np.int64), ref)
    if bits == 8:
        assert ref[0, 0, 0] == 32 * 127 * 127 and ref[-1, -1, -1] == -32 * 127 * 127
    assert qg.device_error() == 0


# ------------------------------------------------------------------ dense products

def _case(M, N, K, bits, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, K)).astype(np.float32)
    x[:, rng.choice(K, max(1, K // 100), replace=False)] *= 20
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    qx, dx = oracle.quantize_act_q8(x)
    qw, dw = oracle.quantize_w_q8_0(w) if bits == 8 else oracle.quantize_w_q4_0(w)
    return qx, dx, qw, dw


GEMV_SHAPES = [(4, 256, 512), (1, 4096, 4096), (3, 200, 96), (8, 1000, 1024), (1, 5, 32),
               (2, 33, 12288), (7, 129, 4160)]
MMA_SHAPES = [(4, 256, 512), (37, 200, 96), (128, 256, 512), (300, 130, 160), (9, 1, 32),
              (513, 384, 1056)]
TC_SHAPES = [(4, 256, 512), (128, 256, 256), (300, 130, 768), (129, 513, 1024), (9, 1, 256),
             (256, 768, 4096), (640, 1000, 2048)]


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("algo,M,N,K", [(qg.ALGO_GEMV,) + s for s in GEMV_SHAPES] +
                         [(qg.ALGO_MMA,) + s for s in MMA_SHAPES] +
                         [(qg.ALGO_TCGEN05,) + s for s in TC_SHAPES])
def test_qgemm_parity(algo, M, N, K, bits):
    qx, dx, qw, dw = _case(M, N, K, bits, M * 7 + N * 3 + K + bits)
    y_ref, mag = oracle.qgemm(qx, dx, qw, dw, bits)
    y = _gemm(bits, algo, to_dev(qx), to_dev(dx), to_dev(qw), to_dev(dw))
    _sync()
    assert_close(to_np(y), y_ref, mag)
    assert qg.device_error() == 0


@pytest.mark.parametrize("bits", [8, 4])
def test_qgemm_tc_whole_tiles_and_split_tail(bits):
    """More 128 x 128 tiles than SMs, a few left over: whole-tile rounds, then the
    leftover tiles (ragged rows and columns) cut along K into chunks whose partial
    sums are added afterwards.  y within tolerance; the same bits on a second run."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n_tiles = sms // 2 + 4
    M, N, K = 200, 128 * n_tiles - 37, 768
    assert (2 * n_tiles) % sms not in (0, 2 * n_tiles)
    qx, dx, qw, dw = _case(M, N, K, bits, 4242 + bits)
    y_ref, mag = oracle.qgemm(qx, dx, qw, dw, bits)
    args = (to_dev(qx), to_dev(dx), to_dev(qw), to_dev(dw))
    y = _gemm(bits, qg.ALGO_TCGEN05, *args)
    _sync()
    assert_close(to_np(y), y_ref, mag)
    assert torch.equal(y, _gemm(bits, qg.ALGO_TCGEN05, *args))
    assert qg.device_error() == 0


@pytest.mark.parametrize("bits", [8, 4])
def test_tc_wait_limit_gives_up_and_recovers(bits):
    """A pipeline wait of the tensor-core kernel that runs out sets the device error
    word, and the call returns (the kernel drains its own copies and MMAs and frees
    tensor memory); the next call on the same GPU is correct.  The wait is made to
    run out by lowering the wait limit to one cycle: nothing is withheld, no trap."""
    M, N, K = 512, 768, 1024
    qx, dx, qw, dw = _case(M, N, K, bits, 777 + bits)
    args = (to_dev(qx), to_dev(dx), to_dev(qw), to_dev(dw))
    assert qg.device_error() == 0
    try:
        qg.debug_set_wait_limit(1)
        for _ in range(3):
            _gemm(bits, qg.ALGO_TCGEN05, *args)
        _sync()
        assert qg.device_error() == 1
    finally:
        qg.debug_set_wait_limit(0)
    y_ref, mag = oracle.qgemm(qx, dx, qw, dw, bits)
    y = _gemm(bits, qg.ALGO_TCGEN05, *args)
    _sync()
    assert qg.device_error() == 0
    assert_close(to_np(y), y_ref, mag)


@pytest.mark.parametrize("pad", [12, 13])            # even / odd ldy (vector / scalar stores)
@pytest.mark.parametrize("algo", DENSE_ALGOS)
def test_qgemm_ldy_and_determinism(algo, pad):
    M, N, K = (4, 300, 640) if algo == qg.ALGO_GEMV else (40, 300, 768)
    qx, dx, qw, dw = _case(M, N, K, 8, 99)
    y_ref, mag = oracle.qgemm(qx, dx, qw, dw, 8)
    big = torch.full((M, N + pad), 7.0, dtype=torch.float32, device=dev())
    args = (to_dev(qx), to_dev(dx), to_dev(qw), to_dev(dw))
    y1 = qg.qgemm_q8_0(*args, y=big[:, :N], algo=algo)
    _sync()
    assert_close(to_np(big[:, :N]), y_ref, mag)
    assert torch.all(big[:, N:] == 7.0)                 # columns past N untouched
    y2 = qg.qgemm_q8_0(*args, algo=algo)
    _sync()
    assert torch.equal(y1, y2)


def test_qgemm_m_zero_is_noop():
    qx = torch.empty((0, 64), dtype=torch.int8, device=dev())
    dx = torch.empty((0, 2), dtype=torch.float32, device=dev())
    qw = torch.zeros((8, 64), dtype=torch.int8, device=dev())
    dw = torch.zeros((8, 2), dtype=torch.float16, device=dev())
    y = qg.qgemm_q8_0(qx, dx, qw, dw)
    assert y.shape == (0, 8)


# ------------------------------------------------------------------ full-size decode

@pytest.fixture(scope="module")
def decode_weights():
    """Q8_0 weights of the four decode projections, quantized by the oracle."""
    out = {}
    for i, (N, K) in enumerate(inputs.DECODE_SHAPES):
        w, x = inputs.decode_case(N, K, M=4, sub=i)
        qw, dw = oracle.quantize_w_q8_0(w)
        out[(N, K)] = (w, x, qw, dw)
    return out


@pytest.mark.parametrize("M", [1, 4])
@pytest.mark.parametrize("shape", inputs.DECODE_SHAPES)
def test_decode_full_shape(decode_weights, shape, M):
    """The decode workload end to end through the ABI (GPU quantizes both
    sides); codes/scales bit-exact on the oracle's, y within tolerance."""
    w, x, qw_ref, dw_ref = decode_weights[shape]
    x = x[:M]
    wt = to_dev(w)
    qw, dw = qg.quantize_weight_q8_0(wt)
    qx, dx = qg.quantize_act_q8(to_dev(x))
    y = qg.qgemm_q8_0(qx, dx, qw, dw)
    _sync()
    del wt
    assert np.array_equal(to_np(qw), qw_ref) and np.array_equal(to_np(dw), dw_ref)
    qx_ref, dx_ref = oracle.quantize_act_q8(x)
    assert np.array_equal(to_np(qx), qx_ref) and np.array_equal(to_np(dx), dx_ref)
    y_ref, mag = oracle.qgemm(qx_ref, dx_ref, qw_ref, dw_ref, 8)
    assert_close(to_np(y), y_ref, mag)


@pytest.mark.parametrize("M", [1, 4])
def test_decode_step_as_benchmarked(M):
    """The decode step exactly as bench.py times it: bench's own buffers and CUDA graphs
    (the one-graph step with dependent launches, the split graphs, the end-to-end graph
    with host copies).  Every projection's output equals a direct call of the ABI bit for
    bit after each replay, and sampled lm-head rows match the oracle."""
    import os
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    projs = bench.make_decode(dev(), M)
    graphs = bench.DecodeGraphs(projs)
    ref = []
    for p in projs:
        qx, dx = qg.quantize_act_q8(p["x"])
        ref.append(qg.qgemm_q8_0(qx, dx, p["qw"], p["dw"]))
    _sync()
    for replay in (graphs.step_full, graphs.step, graphs.step_e2e):
        for p in projs:
            p["y"].fill_(float("nan"))
        replay()
        _sync()
        for p, r in zip(projs, ref):
            assert torch.equal(p["y"], r)
    pk = projs[0]
    host = pk["y_all_host"].clone()
    assert torch.equal(host.to(dev()), pk["y_all"])          # the end-to-end copy out
    p = projs[-1]
    N, K = p["N"], p["K"]
    w, x = inputs.decode_case(N, K, M=M, sub=len(projs) - 1)
    qw_ref, dw_ref = oracle.quantize_w_q8_0(w)
    qx_ref, dx_ref = oracle.quantize_act_q8(x)
    rows = np.sort(np.random.default_rng(11).choice(N, 64, replace=False))
    y_ref, mag = oracle.qgemm(qx_ref, dx_ref, qw_ref[rows], dw_ref[rows], 8)
    assert_close(to_np(p["y"])[:, rows], y_ref, mag)
    del graphs, projs


# ------------------------------------------------------------------ GEMV with the quantization fused

# (M, N, K, x row padding): K-splits W = 1, 2, 4 and 8 among them, a ragged last row
# tile, and rows padded by 3 floats (not 16-byte aligned: scalar x loads); from 8192
# rows at M >= 2 the activations are staged per block (row tiles ragged at N = 8203 and
# 9001)
FUSED_SHAPES = [(1, 4096, 4096, 0), (4, 4096, 4096, 0), (1, 300, 12288, 0), (3, 37, 96, 3),
                (8, 1000, 1024, 0), (2, 33, 12288, 3), (7, 129, 4160, 0), (1, 5, 32, 0),
                (5, 40000, 512, 0), (8, 8203, 1024, 3), (2, 9001, 256, 0), (4, 12288, 4096, 0)]


@pytest.mark.parametrize("M,N,K,pad", FUSED_SHAPES)
def test_fused_gemv_equals_two_launches(M, N, K, pad):
    """qgemv_q8_0_f32(x) writes exactly what quantize_act_q8 + qgemm_q8_0 write, and
    that is within tolerance of the oracle on the oracle's own codes."""
    rng = np.random.default_rng(300 + M * 7 + N + K)
    x = rng.standard_normal((M, K + pad)).astype(np.float32)
    x[0, :32] = 0.0                                   # an all-zero group: d = 0, codes 0
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    qw, dw = qg.quantize_weight_q8_0(to_dev(w))
    xt = to_dev(x)[:, :K]
    y_fused = qg.qgemv_q8_0_f32(xt, qw, dw)
    qx, dx = qg.quantize_act_q8(xt)
    y_two = qg.qgemm_q8_0(qx, dx, qw, dw)
    _sync()
    assert torch.equal(y_fused, y_two)
    qx_ref, dx_ref = oracle.quantize_act_q8(np.ascontiguousarray(x[:, :K]))
    qw_ref, dw_ref = oracle.quantize_w_q8_0(w)
    y_ref, mag = oracle.qgemm(qx_ref, dx_ref, qw_ref, dw_ref, 8)
    assert_close(to_np(y_fused), y_ref, mag)


@pytest.mark.parametrize("M", [1, 4])
def test_fused_gemv_lm_head_full_size(decode_weights, M):
    """The 151936 x 4096 lm-head projection of the decode workload: the fused call
    equals the two-launch path bit for bit; sampled rows against the oracle."""
    shape = inputs.DECODE_SHAPES[-1]
    w, x, qw_ref, dw_ref = decode_weights[shape]
    x = x[:M]
    qw, dw = qg.quantize_weight_q8_0(to_dev(w))
    xt = to_dev(x)
    y_fused = qg.qgemv_q8_0_f32(xt, qw, dw)
    qx, dx = qg.quantize_act_q8(xt)
    y_two = qg.qgemm_q8_0(qx, dx, qw, dw)
    _sync()
    assert torch.equal(y_fused, y_two)
    rows = np.sort(np.random.default_rng(9).choice(shape[0], 64, replace=False))
    qx_ref, dx_ref = oracle.quantize_act_q8(x)
    y_ref, mag = oracle.qgemm(qx_ref, dx_ref, qw_ref[rows], dw_ref[rows], 8)
    assert_close(to_np(y_fused)[:, rows], y_ref, mag)


# ------------------------------------------------------------------ full-size prefill (sampled)

@pytest.mark.parametrize("algo", [qg.ALGO_AUTO, qg.ALGO_MMA])
@pytest.mark.parametrize("shape", inputs.PREFILL_SHAPES)
def test_prefill_full_shape_sampled(shape, algo):
    M, N, K = shape
    i = inputs.PREFILL_SHAPES.index(shape)
    w, x = inputs.prefill_case(M, N, K, sub=i)
    qw, dw = qg.quantize_weight_q8_0(to_dev(w))
    qx, dx = qg.quantize_act_q8(to_dev(x))
    y = qg.qgemm_q8_0(qx, dx, qw, dw, algo=algo)
    _sync()
    assert qg.device_error() == 0
    rows = np.sort(np.random.default_rng(5).choice(M, 12, replace=False))
    rows[-1] = M - 1
    qx_ref, dx_ref = oracle.quantize_act_q8(x[rows])
    qw_ref, dw_ref = oracle.quantize_w_q8_0(w)
    assert np.array_equal(to_np(qw), qw_ref) and np.array_equal(to_np(dw), dw_ref)
    assert np.array_equal(to_np(qx)[rows], qx_ref)
    y_ref, mag = oracle.qgemm(qx_ref, dx_ref, qw_ref, dw_ref, 8)
    assert_close(to_np(y)[rows], y_ref, mag)


# ------------------------------------------------------------------ full-size long context (sampled)

@pytest.mark.parametrize("shape", inputs.LONGCTX_SHAPES)
def test_longctx_full_shape_sampled(shape):
    """M = 18432 through the default path (tensor cores): weights bit-exact on
    sampled rows, y within tolerance on sampled rows, no device error."""
    M, N, K = shape
    i = inputs.LONGCTX_SHAPES.index(shape)
    w, x = inputs.longctx_case(M, N, K, sub=i)
    qw, dw = qg.quantize_weight_q8_0(to_dev(w))
    xt = to_dev(x)
    qx, dx = qg.quantize_act_q8(xt)
    del xt
    y = qg.qgemm_q8_0(qx, dx, qw, dw)
    _sync()
    assert qg.device_error() == 0
    rng = np.random.default_rng(6)
    rows = np.sort(rng.choice(M, 8, replace=False))
    rows[-1] = M - 1
    cols = np.sort(rng.choice(N, 512, replace=False))
    cols[-1] = N - 1
    qw_ref, dw_ref = oracle.quantize_w_q8_0(w[cols])
    assert np.array_equal(to_np(qw[torch.from_numpy(cols).to(dev())]), qw_ref)
    qx_ref, dx_ref = oracle.quantize_act_q8(x[rows])
    assert np.array_equal(to_np(qx)[rows], qx_ref)
    y_ref, mag = oracle.qgemm(qx_ref, dx_ref, qw_ref, dw_ref, 8)
    yg = to_np(y[torch.from_numpy(rows).to(dev())])[:, cols]
    assert_close(yg, y_ref, mag)


# ------------------------------------------------------------------ MoE

def _moe_small(E=9, T=53, topk=3, N=96, K=128, seed=3):
    rng = np.random.default_rng(seed)
    w = (rng.standard_normal((E, N, K)) * 0.02).astype(np.float32)
    qw4 = np.empty((E, N, K // 2), np.uint8)
    dw = np.empty((E, N, K // 32), np.uint16)
    for e in range(E):
        qw4[e], dw[e] = oracle.quantize_w_q4_0(w[e])
    ids = inputs.zipf_routing(rng, T, E, topk)
    return rng, qw4, dw, ids


@pytest.mark.parametrize("E,T,topk", [(9, 53, 3), (128, 947, 8), (1024, 300, 4), (5, 1, 1)])
def test_moe_route_bit_exact(E, T, topk):
    rng = np.random.default_rng(E + T)
    ids = inputs.zipf_routing(rng, T, E, topk)
    counts, offsets, perm, bad = oracle.moe_route(ids, E)
    c, o, p, d_err = qg.moe_route(to_dev(ids), E)
    _sync()
    assert bad == 0 and int(to_np(d_err)[0]) == 0
    assert np.array_equal(to_np(c), counts)
    assert np.array_equal(to_np(o), offsets)
    assert np.array_equal(to_np(p)[: offsets[E]], perm)


def test_moe_route_invalid_ids():
    ids = np.array([[0, 5], [7, 1], [-1, 0], [3, 3]], np.int32)
    counts, offsets, perm, bad = oracle.moe_route(ids, 6)
    c, o, p, d_err = qg.moe_route(to_dev(ids), 6)
    _sync()
    assert int(to_np(d_err)[0]) == bad == 2
    assert np.array_equal(to_np(c), counts) and np.array_equal(to_np(o), offsets)
    assert np.array_equal(to_np(p)[: offsets[6]], perm)


def test_moe_empty_batch():
    """No tokens: routing writes all-zero counts and offsets, the grouped product returns
    an empty output and flags nothing."""
    ids = torch.empty((0, 8), dtype=torch.int32, device=dev())
    c, o, p, d_err = qg.moe_route(ids, 16)
    _sync()
    assert np.all(to_np(c) == 0) and np.all(to_np(o) == 0) and int(to_np(d_err)[0]) == 0
    E, N, K = 4, 64, 256
    qw4 = torch.zeros((E, N, K // 2), dtype=torch.uint8, device=dev())
    dw = torch.zeros((E, N, K // 32), dtype=torch.float16, device=dev())
    qx = torch.zeros((0, K), dtype=torch.int8, device=dev())
    dx = torch.zeros((0, K // 32), dtype=torch.float32, device=dev())
    y, err = qg.grouped_qgemm_moe(qx, dx, torch.empty((0, 2), dtype=torch.int32, device=dev()),
                                  0, qw4, dw)
    _sync()
    assert y.shape == (0, N) and int(to_np(err)[0]) == 0 and qg.device_error() == 0


@pytest.mark.parametrize("K", [128, 512])      # K % 256 == 0 takes the tensor-core kernel
@pytest.mark.parametrize("mode", [0, 1])
def test_grouped_moe_small(mode, K):
    rng, qw4, dw, ids = _moe_small(K=K)
    T, topk = ids.shape
    rows = T if mode == 0 else T * topk
    x = rng.standard_normal((rows, K)).astype(np.float32)
    qx, dx = oracle.quantize_act_q8(x)
    y_ref, mag, bad = oracle.grouped_qgemm_moe(qx, dx, ids, mode, qw4, dw)
    y, d_err = qg.grouped_qgemm_moe(to_dev(qx), to_dev(dx), to_dev(ids), mode, to_dev(qw4),
                                    to_dev(dw))
    _sync()
    assert bad == 0 and int(to_np(d_err)[0]) == 0
    assert_close(to_np(y), y_ref, mag)


def _replay_in_graph(call):
    """Capture call() in a CUDA graph (after one eager run on a side stream, which
    capture needs) and replay it twice."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    return g


@pytest.mark.parametrize("bits", [8, 4])
def test_tc_dense_call_replays_in_cuda_graph(bits):
    """A tensor-core product is a chain of programmatic dependent launches (pre-pass,
    GEMM, tail reduction); captured in a CUDA graph the chain becomes graph edges, and
    every replay gives the eager result bit for bit."""
    M, N, K = 300, 520, 1024
    qx, dx, qw, dw = _case(M, N, K, bits, 9090 + bits)
    args = (to_dev(qx), to_dev(dx), to_dev(qw), to_dev(dw))
    y_eager = _gemm(bits, qg.ALGO_TCGEN05, *args)
    _sync()
    y = torch.empty_like(y_eager)
    g = _replay_in_graph(lambda: _gemm(bits, qg.ALGO_TCGEN05, *args, y=y))
    for _ in range(2):
        y.fill_(float("nan"))
        g.replay()
        _sync()
        assert torch.equal(y, y_eager)
    assert qg.device_error() == 0


@pytest.mark.parametrize("mode", [0, 1])
def test_grouped_moe_replays_in_cuda_graph(mode):
    """The grouped product (routing with its tile table, gather, tensor-core GEMM) in a
    CUDA graph: every replay gives the eager result bit for bit."""
    rng, qw4, dw, ids = _moe_small(K=512)
    T, topk = ids.shape
    rows = T if mode == 0 else T * topk
    qx, dx = oracle.quantize_act_q8(rng.standard_normal((rows, 512)).astype(np.float32))
    a = (to_dev(qx), to_dev(dx), to_dev(ids), mode, to_dev(qw4), to_dev(dw))
    y_eager, _ = qg.grouped_qgemm_moe(*a)
    _sync()
    y = torch.empty_like(y_eager)
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    g = _replay_in_graph(lambda: qg.grouped_qgemm_moe(*a, y=y, d_err=err))
    for _ in range(2):
        y.fill_(float("nan"))
        g.replay()
        _sync()
        assert torch.equal(y, y_eager)
    assert int(to_np(err)[0]) == 0 and qg.device_error() == 0


def test_tc_chains_on_a_side_stream():
    """The programmatic dependent launches of a call stay on the caller's stream: the
    tensor-core dense and grouped products issued on a side stream, right after work
    that writes their inputs on that stream, equal the default-stream results."""
    M, N, K = 200, 384, 1024
    qx, dx, qw, dw = _case(M, N, K, 8, 4711)
    args = (to_dev(qx), to_dev(dx), to_dev(qw), to_dev(dw))
    y_ref = _gemm(8, qg.ALGO_TCGEN05, *args)
    rng, qw4, dw4, ids = _moe_small(K=512)
    qx2, dx2 = oracle.quantize_act_q8(rng.standard_normal((ids.shape[0], 512)).astype(np.float32))
    a = (to_dev(qx2), to_dev(dx2), to_dev(ids), 0, to_dev(qw4), to_dev(dw4))
    ym_ref, _ = qg.grouped_qgemm_moe(*a)
    _sync()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        qx_s = torch.empty_like(args[0])
        qx_s.copy_(args[0])                          # the input is written on the side stream
        y = _gemm(8, qg.ALGO_TCGEN05, qx_s, *args[1:])
        ym, err = qg.grouped_qgemm_moe(*a)
    torch.cuda.current_stream().wait_stream(side)
    _sync()
    assert torch.equal(y, y_ref) and torch.equal(ym, ym_ref)
    assert int(to_np(err)[0]) == 0 and qg.device_error() == 0


@pytest.mark.parametrize("K", [128, 256])
def test_grouped_moe_unrouted_rows_zero_and_counted(K):
    rng, qw4, dw, ids = _moe_small(K=K)
    ids = ids.copy()
    ids[4, 1] = 9          # == E: out of range
    ids[10, 0] = -2
    x = rng.standard_normal((ids.shape[0], K)).astype(np.float32)
    qx, dx = oracle.quantize_act_q8(x)
    y_ref, mag, bad = oracle.grouped_qgemm_moe(qx, dx, ids, 0, qw4, dw)
    y0 = torch.full((ids.size, 96), 5.0, device=dev())
    y, d_err = qg.grouped_qgemm_moe(to_dev(qx), to_dev(dx), to_dev(ids), 0, to_dev(qw4),
                                    to_dev(dw), y=y0)
    _sync()
    assert bad == 2 and int(to_np(d_err)[0]) == 2
    assert_close(to_np(y), y_ref, mag)


@pytest.mark.parametrize("K,algo", [(128, qg.ALGO_MMA), (256, qg.ALGO_TCGEN05),
                                     (512, qg.ALGO_TCGEN05)])
def test_grouped_moe_single_expert_equals_dense_q4(K, algo):
    """Every row routed to one expert: the MoE product is the dense product of that
    expert's weights.  Bit for bit where both add the groups in the same order (the
    MMA kernels; the tensor-core kernels at 8 groups, which the dense kernel never
    cuts along K).  At 16 groups the dense kernel's 3 tiles, fewer than the SMs, are
    each summed as two K chunks, so both products are held to the oracle instead."""
    rng, qw4, dw, _ = _moe_small(K=K)
    T = 300
    ids = np.full((T, 1), 6, np.int32)
    x = rng.standard_normal((T, K)).astype(np.float32)
    qx, dx = qg.quantize_act_q8(to_dev(x))
    y, _ = qg.grouped_qgemm_moe(qx, dx, to_dev(ids), 0, to_dev(qw4), to_dev(dw))
    yd = qg.qgemm_q4_0(qx, dx, to_dev(qw4[6]), to_dev(dw[6]), algo=algo)
    _sync()
    if K == 512:
        y_ref, mag = oracle.qgemm(to_np(qx), to_np(dx), qw4[6], dw[6], 4)
        assert_close(to_np(y), y_ref, mag)
        assert_close(to_np(yd), y_ref, mag)
    else:
        assert torch.equal(y, yd)


@pytest.fixture(scope="module")
def moe_full():
    return inputs.moe_case()


@pytest.mark.parametrize("which", ["gate_up", "down"])
def test_grouped_moe_full_config_sampled(moe_full, which):
    d = moe_full
    ids = d["topk_ids"]
    E = ids.max() + 1
    if which == "gate_up":
        w, x, mode = d["w_gate_up"], d["x_tok"], 0
    else:
        w, x, mode = d["w_down"], d["x_pair"], 1
    E, N, K = w.shape
    wt = to_dev(w.reshape(E * N, K))
    qw4, dw = qg.quantize_weight_q4_0(wt)
    del wt
    qw4 = qw4.view(E, N, K // 2)
    dw = dw.view(E, N, K // 32)
    qx, dx = qg.quantize_act_q8(to_dev(x))
    y, d_err = qg.grouped_qgemm_moe(qx, dx, to_dev(ids), mode, qw4, dw)
    _sync()
    assert int(to_np(d_err)[0]) == 0
    rng = np.random.default_rng(8)
    P = ids.size
    pairs = rng.choice(P, 48, replace=False)
    flat = ids.ravel()
    # the busiest expert's rows are included
    busiest = np.bincount(flat, minlength=E).argmax()
    pairs = np.concatenate([pairs, np.nonzero(flat == busiest)[0][-4:]])
    yg = to_np(y)
    qw4_np, dw_np = to_np(qw4), to_np(dw)
    for e in np.unique(flat[pairs]):
        q_ref, d_ref = oracle.quantize_w_q4_0(w[e])
        assert np.array_equal(qw4_np[e], q_ref) and np.array_equal(dw_np[e], d_ref)
        sel = pairs[flat[pairs] == e]
        xr = sel // 8 if mode == 0 else sel
        qx_ref, dx_ref = oracle.quantize_act_q8(x[xr])
        y_ref, mag = oracle.qgemm(qx_ref, dx_ref, q_ref, d_ref, 4)
        assert_close(yg[sel], y_ref, mag)


# ------------------------------------------------------------------ MoE steps around the GEMM

def _swiglu_reference_check(gu: np.ndarray, F: int, qh: np.ndarray, dh: np.ndarray):
    """qh/dh against the binary64 SwiGLU: scales within binary32 rounding, codes the
    round-half-even of h / d except within 1e-4 of a half-integer, where either
    neighbour is a correct result of a binary32 evaluation."""
    h = oracle.silu_mul(gu, F)
    P = h.shape[0]
    hg = h.reshape(P, F // 32, 32)
    d_ref = np.abs(hg).max(axis=2) / 127.0
    assert np.allclose(dh, d_ref, rtol=1e-6, atol=0.0)
    zero = d_ref == 0
    assert np.all(dh[zero] == 0)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(zero[:, :, None], 0.0, hg / d_ref[:, :, None])
    q_ref = np.clip(np.rint(r), -127, 127)
    frac = np.abs(np.abs(r) - np.floor(np.abs(r)) - 0.5)
    near = frac < 1e-4
    qg_ = qh.reshape(P, F // 32, 32).astype(np.float64)
    assert np.array_equal(qg_[~near], q_ref[~near])
    assert np.all(np.abs(qg_[near] - r[near]) <= 0.5 + 1e-4)
    return int(near.sum())


@pytest.mark.parametrize("P,F,pad", [(300, 1024, 0), (37, 96, 40), (1, 32, 0)])
def test_swiglu_quant_vs_oracle(P, F, pad):
    rng = np.random.default_rng(7 + P + F)
    gu = (rng.standard_normal((P, 2 * F + pad)) * 2.0).astype(np.float32)
    gu[0, :32] = 0.0                                   # gate 0: h = 0, d = 0, q = 0
    if P > 1:
        gu[-1, :4] = [40.0, -40.0, 88.0, -88.0]        # saturated and vanishing gates
    gu_t = to_dev(gu)
    qh, dh = qg.moe_swiglu_quant(gu_t, F)
    _sync()
    _swiglu_reference_check(gu, F, to_np(qh), to_np(dh))
    assert np.all(to_np(qh)[0, :32] == 0) and to_np(dh)[0, 0] == 0.0


@pytest.mark.parametrize("T,topk,N", [(947, 8, 2048), (13, 3, 1030), (1, 1, 4)])
def test_moe_combine_vs_oracle(T, topk, N):
    rng = np.random.default_rng(11 + T + N)
    y = rng.standard_normal((T * topk, N)).astype(np.float32)
    y[0] = 0.0                                         # an unrouted pair's zero row
    w = rng.random((T, topk)).astype(np.float32)
    w /= w.sum(axis=1, keepdims=True)
    out = qg.moe_combine(to_dev(y), to_dev(w))
    _sync()
    ref, mag = oracle.moe_combine(y, w)
    err = np.abs(to_np(out).astype(np.float64) - ref)
    assert np.all(err <= 1e-6 * mag + 1e-30)
    out2 = qg.moe_combine(to_dev(y), to_dev(w))         # deterministic slot order
    _sync()
    assert torch.equal(out, out2)


def test_moe_layer_end_to_end():
    """gate/up -> SwiGLU + re-quantization -> down -> router-weighted combine, all on the
    GPU through the C ABI, against the oracle's composition of the same steps."""
    E, T, topk, F, K = 16, 96, 4, 256, 256
    rng = np.random.default_rng(2026)
    wgu = (rng.standard_normal((E, 2 * F, K)) * 0.02).astype(np.float32)
    wdn = (rng.standard_normal((E, K, F)) * 0.02).astype(np.float32)
    qgu = np.empty((E, 2 * F, K // 2), np.uint8)
    dgu = np.empty((E, 2 * F, K // 32), np.uint16)
    qdn = np.empty((E, K, F // 2), np.uint8)
    ddn = np.empty((E, K, F // 32), np.uint16)
    for e in range(E):
        qgu[e], dgu[e] = oracle.quantize_w_q4_0(wgu[e])
        qdn[e], ddn[e] = oracle.quantize_w_q4_0(wdn[e])
    ids = inputs.zipf_routing(rng, T, E, topk)
    x = rng.standard_normal((T, K)).astype(np.float32)
    w = rng.random((T, topk)).astype(np.float32)
    w /= w.sum(axis=1, keepdims=True)
    qx, dx = oracle.quantize_act_q8(x)
    # oracle composition
    gu_ref, _, _ = oracle.grouped_qgemm_moe(qx, dx, ids, 0, qgu, dgu)
    qh_ref, dh_ref = oracle.quantize_act_q8(oracle.silu_mul(gu_ref, F).astype(np.float32))
    yd_ref, yd_mag, _ = oracle.grouped_qgemm_moe(qh_ref, dh_ref, ids, 1, qdn, ddn)
    out_ref, out_mag = oracle.moe_combine(yd_ref, w)
    # GPU
    gu, _ = qg.grouped_qgemm_moe(to_dev(qx), to_dev(dx), to_dev(ids), 0, to_dev(qgu), to_dev(dgu))
    qh, dh = qg.moe_swiglu_quant(gu, F)
    yd, _ = qg.grouped_qgemm_moe(qh, dh, to_dev(ids), 1, to_dev(qdn), to_dev(ddn))
    out = qg.moe_combine(yd, to_dev(w))
    _sync()
    qh_np = to_np(qh)
    flip = qh_np != qh_ref
    assert int(flip.sum()) <= qh_ref.size // 1000    # codes differ only at near-ties
    assert np.all(np.abs(qh_np.astype(np.int32) - qh_ref.astype(np.int32))[flip] == 1)
    # A code flipped by one in pair row p, group g moves y_down[p, n] by at most
    # dh[p, g] * dw[e(p), n, g] * max|q4| (|q4| <= 8); only the tokens holding
    # such a pair get that extra allowance, every other token keeps the 1e-5 bar.
    dwn = oracle.f16_bits_to_f32(ddn).astype(np.float64).reshape(ddn.shape)   # [E, K, F/32]
    dh_hi = np.maximum(to_np(dh), dh_ref).astype(np.float64)   # either side's group scale
    extra = np.zeros((T * topk, K))
    for p, k in zip(*np.nonzero(flip)):
        g = k // 32
        extra[p] += dh_hi[p, g] * dwn[ids.reshape(-1)[p], :, g] * 8.0
    wsum = np.abs(w[:, :, None].astype(np.float64) * yd_mag.reshape(T, topk, K)).sum(1)
    wextra = (w[:, :, None].astype(np.float64) * extra.reshape(T, topk, K)).sum(1)
    err = np.abs(to_np(out).astype(np.float64) - out_ref)
    assert np.all(err <= 1e-5 * wsum + wextra + 1e-30)


# ------------------------------------------------------------------ GGUF block import

# block counts 111, 38400 and 38528 (a multiple of 256 and not); off = 2: the input
# 2 bytes past 16-byte alignment (the format only guarantees 2-byte alignment)
@pytest.mark.parametrize("wbits", [8, 4])
@pytest.mark.parametrize("N,K,off", [(37, 96, 0), (300, 4096, 0), (301, 4096, 0), (301, 4096, 2)])
def test_gguf_import_bit_exact(wbits, N, K, off):
    """The CUDA import equals the oracle byte for byte, and the imported weights give
    the same product as the same weights quantized planar."""
    rng = np.random.default_rng(90 + N + wbits)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    q, d = oracle.quantize_w_q8_0(w) if wbits == 8 else oracle.quantize_w_q4_0(w)
    cb = 32 if wbits == 8 else 16
    G = K // 32
    blocks = np.empty((N, G, 2 + cb), np.uint8)
    blocks[:, :, 0] = (d & 0xFF).astype(np.uint8)
    blocks[:, :, 1] = (d >> 8).astype(np.uint8)
    blocks[:, :, 2:] = q.view(np.uint8).reshape(N, G, cb)
    imp = qg.import_gguf_q8_0 if wbits == 8 else qg.import_gguf_q4_0
    flat = blocks.reshape(-1)
    buf = torch.zeros(flat.size + off, dtype=torch.uint8, device="cuda")
    buf[off:].copy_(to_dev(flat))
    qt, dt = imp(buf[off:], N, K)
    _sync()
    q_ref, d_ref = oracle.import_gguf(blocks.reshape(-1), N, K, wbits)
    assert np.array_equal(to_np(qt).view(np.uint8), q_ref.view(np.uint8))
    assert np.array_equal(to_np(dt).view(np.uint16), d_ref)


# ------------------------------------------------------------------ split-K attention merge

@pytest.mark.parametrize("S,R,D", [(1, 5, 128), (4, 300, 128), (64, 37, 100), (7, 1024, 256)])
def test_splitk_merge_vs_oracle(S, R, D):
    rng = np.random.default_rng(500 + S + R + D)
    m = (rng.standard_normal((S, R)) * 4.0).astype(np.float32)
    l = (rng.random((S, R)) * 30.0 + 1.0).astype(np.float32)
    acc = (rng.standard_normal((S, R, D)) * l[:, :, None]).astype(np.float32)
    if S > 1:
        m[1, :R // 2] = -np.inf                             # empty splits
        l[1, :R // 2] = 0.0
        acc[1, :R // 2] = 0.0
        m[:, -1] = -np.inf                                  # a row with no key at all
        l[:, -1] = 0.0
        acc[:, -1] = 0.0
    out, lse = qg.attn_splitk_merge(to_dev(m), to_dev(l), to_dev(acc))
    _sync()
    ref, ref_lse, mag = oracle.splitk_merge(m, l, acc)
    o = to_np(out).astype(np.float64)
    assert np.all(np.abs(o - ref) <= 2e-6 * mag + 1e-30)
    ls = to_np(lse).astype(np.float64)
    fin = np.isfinite(ref_lse)
    assert np.all(np.abs(ls[fin] - ref_lse[fin]) <= 1e-6 * np.maximum(1.0, np.abs(ref_lse[fin])))
    assert np.all(ls[~fin] == -np.inf) and np.all(o[~fin] == 0.0)
    out2, _ = qg.attn_splitk_merge(to_dev(m), to_dev(l), to_dev(acc))
    _sync()
    assert torch.equal(out, out2)


# ------------------------------------------------------------------ 3-bit WHT + Lloyd-Max KV codec

def _kv3_codes(codes, D):
    E = D // 32
    c = codes.view(np.uint32).astype(np.int64)
    k = np.zeros((c.shape[0], D), np.int64)
    for j in range(D):
        L, e = divmod(j, E)
        for b in range(3):
            k[:, j] |= ((c[:, b * E + e] >> L) & 1) << b
    return k


# (row stride, row offset): 16-byte rows take the vector path, the others the scalar one;
# T not a multiple of the vectors a warp takes per step (32 / (D / 32))
@pytest.mark.parametrize("T,D,pad,off", [(1000, 128, 0, 0), (333, 64, 16, 0), (257, 256, 0, 0),
                                         (201, 128, 3, 0), (129, 64, 5, 1), (77, 256, 4, 2)])
def test_kv3_encode_vs_oracle(T, D, pad, off):
    """Scales within binary32 rounding of the binary64 oracle; codes identical except where
    y / s lies within 1e-5 of a decision threshold."""
    rng = np.random.default_rng(600 + T + D)
    x = (rng.standard_normal((T, D + pad)) * rng.uniform(0.01, 10.0, (T, 1))).astype(np.float32)
    x[0] = 0.0
    xt = to_dev(x)[:, off:off + D]
    codes, scales = qg.kv3_encode(xt)
    _sync()
    oc, osc, u = oracle.kv3_encode(np.ascontiguousarray(x[:, off:off + D]))
    sc = to_np(scales).astype(np.float64)
    assert np.all(np.abs(sc - osc) <= 4e-7 * osc)
    kg, ko = _kv3_codes(to_np(codes), D), _kv3_codes(oc, D)
    _, th = oracle.kv3_codebook()
    near = np.min(np.abs(u[:, :, None] - th[None, None, :].astype(np.float32)), axis=2) < 1e-5
    assert np.array_equal(kg[~near], ko[~near])
    assert np.all(np.abs(kg[near] - ko[near]) <= 1)
    assert np.all(kg[0] == 0) and sc[0] == 0.0


@pytest.mark.parametrize("T,D", [(1000, 128), (77, 64), (300, 256)])
def test_kv3_decode_vs_oracle(T, D):
    """Decoding arbitrary codes and scales matches the binary64 oracle to binary32 rounding."""
    rng = np.random.default_rng(700 + T + D)
    codes = rng.integers(0, 2 ** 32, (T, 3 * D // 32), dtype=np.uint64).astype(np.uint32)
    scales = (rng.random(T) * 5.0).astype(np.float32)
    x = qg.kv3_decode(to_dev(codes.view(np.int32)), to_dev(scales), D)
    _sync()
    ref = oracle.kv3_decode(codes, scales, D)
    bound = 1e-6 * scales[:, None].astype(np.float64) * 2.2 * np.sqrt(D) + 1e-30
    assert np.all(np.abs(to_np(x).astype(np.float64) - ref) <= bound)


@pytest.mark.parametrize("T,D,pad,off", [(97, 128, 3, 1), (65, 64, 2, 0), (33, 256, 5, 3)])
def test_kv3_decode_unaligned(T, D, pad, off):
    """Code words one word off 16-byte alignment and strided, unaligned output rows (the
    scalar paths) decode like the aligned call; round trip of an encode stays close."""
    rng = np.random.default_rng(800 + T + D)
    W = 3 * D // 32
    codes = rng.integers(0, 2 ** 32, (T, W), dtype=np.uint64).astype(np.uint32)
    scales = (rng.random(T) * 5.0).astype(np.float32)
    flat = torch.zeros(T * W + 1, dtype=torch.int32, device="cuda")
    cview = flat[1:].view(T, W)
    cview.copy_(to_dev(codes.view(np.int32)))
    big = torch.full((T, D + pad), -7.0, device="cuda")
    out = big[:, off:off + D]
    qg.kv3_decode(cview, to_dev(scales), D, out=out)
    aligned = qg.kv3_decode(to_dev(codes.view(np.int32)), to_dev(scales), D)
    _sync()
    assert torch.equal(out, aligned)
    keep = torch.ones(D + pad, dtype=torch.bool)
    keep[off:off + D] = False
    assert torch.all(big[:, keep.cuda()] == -7.0)
    ref = oracle.kv3_decode(codes, scales, D)
    bound = 1e-6 * scales[:, None].astype(np.float64) * 2.2 * np.sqrt(D) + 1e-30
    assert np.all(np.abs(to_np(out).astype(np.float64) - ref) <= bound)
