"""Pins of the CPU oracle against facts fixed outside it.

Nothing here re-types the oracle's own formulas: each test checks the oracle
against numpy's IEEE binary16 conversion, hand-derived fixtures under
tests/golden/, closed forms, a brute-force dequantized float64 matmul written
with numpy, pure-Python integer dot products, or invariants of the method.
The method: Q8_0 / Q4_0 block quantization in groups of 32 along K with
y[m,n] = sum_g dw[n,g] dx[m,g] S[m,n,g] ("I wrote a custom CUDA inference engine
to run Qwen3.5-27B on a $130 mining card" -- Features; "A 35B Hybrid-Attention
Mixture-of-Experts Model on a 6GB 2011 GPU" -- Methodology 1 and 2).
"""
import os

import numpy as np
import pytest

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _read_pairs(name):
    head, rows = {}, []
    for line in open(os.path.join(GOLD, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        parts = line.split()
        if parts[0] in ("d", "dbits", "w", "q", "bytes"):
            head[parts[0]] = parts[1:]
        else:
            rows.append((float(parts[0]), int(parts[1])))
    return head, rows


# ---------------------------------------------------------------- binary16

def test_f16_encode_matches_numpy():
    rng = np.random.default_rng(7)
    specials = np.array([0.0, -0.0, 1.0, -1.0, 65504.0, 65519.99, 65520.0, 65536.0, 1e9,
                         2.0 ** -14, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -26,
                         2.0 ** -14 - 2.0 ** -25, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11,
                         np.inf, -np.inf], dtype=np.float32)
    rand = np.concatenate([
        rng.standard_normal(3000).astype(np.float32) * np.float32(0.01),
        (rng.standard_normal(3000) * 1e4).astype(np.float32),
        np.exp(rng.uniform(-20, 12, 3000)).astype(np.float32),
        # exact ties between neighbouring binary16 values
        ((np.arange(1, 2048, 3, dtype=np.float64) + 0.5) * 2.0 ** -24).astype(np.float32),
        ((np.arange(1024, 2048, 3, dtype=np.float64) + 0.5) * 2.0 ** -6).astype(np.float32),
    ])
    v = np.concatenate([specials, rand, -rand])
    got = oracle.f32_to_f16_bits(v)
    with np.errstate(over="ignore"):
        want = v.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want)


def test_f16_decode_all_patterns():
    bits = np.arange(65536, dtype=np.uint16)
    want = bits.view(np.float16).astype(np.float32)
    got = oracle.f16_bits_to_f32(bits)
    finite = np.isfinite(want)
    assert np.array_equal(got[finite].view(np.uint32), want[finite].view(np.uint32))
    assert np.array_equal(np.isnan(got), np.isnan(want))
    assert np.array_equal(np.isinf(got), np.isinf(want))


# ---------------------------------------------------------------- activations

@pytest.mark.parametrize("name", ["q8_act_ties.txt", "q8_act_half.txt"])
def test_act_golden(name):
    head, rows = _read_pairs(name)
    x = np.array([r[0] for r in rows], np.float32)[None, :]
    qx, dx = oracle.quantize_act_q8(x)
    assert dx[0, 0] == np.float32(float(head["d"][0]))
    assert qx[0].tolist() == [r[1] for r in rows]


def _act_data(seed=1, M=17, K=256):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, K)).astype(np.float32)
    x[:, rng.choice(K, 5, replace=False)] *= 30
    x[M - 1, :32] = 0.0                               # a zero group
    x[0, 32:64] = np.float32(1e-3) * x[0, 32:64]       # a small-scale group
    return x


def test_act_roundtrip_bound_and_range():
    x = _act_data()
    qx, dx = oracle.quantize_act_q8(x)
    M, K = x.shape
    d = np.repeat(dx.astype(np.float64), 32, axis=1)
    err = np.abs(x.astype(np.float64) - d * qx)
    assert np.all(err <= d * (0.5 + 2.0 ** -16))
    assert np.all(np.abs(qx.astype(np.int32)) <= 127)
    amax = np.abs(x).reshape(M, K // 32, 32).max(axis=2)
    qmax = np.abs(qx.astype(np.int32)).reshape(M, K // 32, 32).max(axis=2)
    assert np.all(qmax[amax > 0] == 127)
    assert np.all(qmax[amax == 0] == 0) and np.all(dx[amax == 0] == 0)
    # the scale is the binary32 quotient max|x| / 127
    assert np.array_equal(dx, (amax / np.float32(127.0)).astype(np.float32))


def test_act_odd_symmetry():
    x = _act_data(2)
    q1, d1 = oracle.quantize_act_q8(x)
    q2, d2 = oracle.quantize_act_q8(-x)
    assert np.array_equal(q2, -q1) and np.array_equal(d1, d2)


@pytest.mark.parametrize("k", [-12, -3, 1, 7, 20])
def test_act_power_of_two_invariance(k):
    x = _act_data(3)
    q1, d1 = oracle.quantize_act_q8(x)
    q2, d2 = oracle.quantize_act_q8(x * np.float32(2.0 ** k))
    assert np.array_equal(q1, q2)
    assert np.array_equal(d2, d1 * np.float32(2.0 ** k))


def test_act_subnormal_scales():
    # max|x| so small that max|x|/127 underflows to 0 -> q = 0; slightly larger
    # max|x| gives a subnormal d and q still follows q = rhe(x/d) clamped.
    tiny = np.float32(2.0 ** -149)
    x = np.zeros((2, 32), np.float32)
    x[0, :3] = [tiny, -tiny, 3 * tiny]
    x[1, :4] = [200 * tiny, -100 * tiny, 50 * tiny, 0]
    qx, dx = oracle.quantize_act_q8(x)
    assert dx[0, 0] == 0 and np.all(qx[0] == 0)
    assert dx[1, 0] == np.float32(2 * tiny)            # rn(200/127) = 2 units
    assert qx[1, :4].tolist() == [100, -50, 25, 0]


# ---------------------------------------------------------------- weights

def test_q8_weight_golden():
    head, rows = _read_pairs("q8_weight_pow2.txt")
    w = (np.array([r[0] for r in rows], np.float64) / 256.0).astype(np.float32)[None, :]
    qw, dw = oracle.quantize_w_q8_0(w)
    assert dw[0, 0] == int(head["dbits"][0], 16)
    assert qw[0].tolist() == [r[1] for r in rows]


def test_q4_pack_golden():
    head, _ = _read_pairs("q4_pack.txt")
    w = np.array([float(t) for t in head["w"]], np.float32)[None, :]
    qw4, dw = oracle.quantize_w_q4_0(w)
    assert dw[0, 0] == int(head["dbits"][0], 16)
    assert qw4[0].tolist() == [int(b, 16) for b in head["bytes"]]


def _unpack_q4(qw4):
    """numpy unpack of the nibble layout: byte j -> element j (low), j+16 (high)."""
    N, half = qw4.shape
    b = qw4.reshape(N, half // 16, 16)
    lo = (b & 0x0F).astype(np.int32) - 8
    hi = (b >> 4).astype(np.int32) - 8
    return np.concatenate([lo, hi], axis=2).reshape(N, half * 2)


def _weights(seed=5, N=23, K=192, std=0.02):
    rng = np.random.default_rng(seed)
    w = (rng.standard_normal((N, K)) * std).astype(np.float32)
    w[2, :32] = 0.0
    return w


@pytest.mark.parametrize("bits,qmax", [(8, 127), (4, 7)])
def test_weight_roundtrip_bound(bits, qmax):
    w = _weights()
    N, K = w.shape
    if bits == 8:
        qw, dw = oracle.quantize_w_q8_0(w)
        q = qw.astype(np.int32)
    else:
        qw4, dw = oracle.quantize_w_q4_0(w)
        q = _unpack_q4(qw4)
    d16 = np.repeat(dw.view(np.float16).astype(np.float64), 32, axis=1)
    assert np.all(np.abs(w - d16 * q) <= d16 * (0.5 + 2.0 ** -16))
    amax = np.abs(w).reshape(N, K // 32, 32).max(axis=2)
    # the stored scale is the binary16 rounding of the binary32 quotient
    want = (amax / np.float32(qmax)).astype(np.float32).astype(np.float16).view(np.uint16)
    assert np.array_equal(dw, want)
    qabs = np.abs(q).reshape(N, K // 32, 32).max(axis=2)
    assert np.all(qabs[amax > 0] == qmax) and np.all(qabs[amax == 0] == 0)
    assert q.min() >= -qmax and q.max() <= qmax      # symmetric: -8 never produced


def test_weight_scale_saturates():
    w = np.zeros((1, 32), np.float32)
    w[0, 0] = 1e8                                     # 1e8/127 > 65504
    qw, dw = oracle.quantize_w_q8_0(w)
    assert dw[0, 0] == 0x7BFF and qw[0, 0] == 127


# ---------------------------------------------------------------- group dots

def _brute_dots(qx, qwv, K):
    M, N = qx.shape[0], qwv.shape[0]
    S = np.zeros((M, N, K // 32), np.int64)
    for m in range(M):
        for n in range(N):
            for g in range(K // 32):
                S[m, n, g] = sum(int(qx[m, k]) * int(qwv[n, k]) for k in range(g * 32, g * 32 + 32))
    return S


def test_group_dots_q8_bruteforce_and_bounds():
    rng = np.random.default_rng(11)
    qx = rng.integers(-127, 128, (3, 96)).astype(np.int8)
    qw = rng.integers(-127, 128, (5, 96)).astype(np.int8)
    qx[0, :32] = 127
    qw[0, :32] = -127
    S = oracle.group_dots(qx, qw, 96, 8)
    assert np.array_equal(S, _brute_dots(qx, qw, 96))
    assert S[0, 0, 0] == -32 * 127 * 127
    assert np.abs(S).max() <= 32 * 127 * 127
    # permuting the elements inside each group leaves S unchanged
    perm = np.concatenate([g * 32 + rng.permutation(32) for g in range(3)])
    assert np.array_equal(oracle.group_dots(qx[:, perm], qw[:, perm], 96, 8), S)


def test_group_dots_q4_bruteforce():
    rng = np.random.default_rng(12)
    qx = rng.integers(-127, 128, (2, 64)).astype(np.int8)
    qw4 = rng.integers(0, 256, (4, 32)).astype(np.uint8)
    S = oracle.group_dots(qx, qw4, 64, 4)
    assert np.array_equal(S, _brute_dots(qx, _unpack_q4(qw4), 64))
    assert np.abs(S).max() <= 32 * 127 * 8


# ---------------------------------------------------------------- products

def _dequant_matmul(qx, dx, qwv, dw):
    """float64 dequantized matmul written with numpy (independent decode of dw)."""
    xd = qx.astype(np.float64) * np.repeat(dx.astype(np.float64), 32, axis=1)
    wd = qwv.astype(np.float64) * np.repeat(dw.view(np.float16).astype(np.float64), 32, axis=1)
    return xd @ wd.T


@pytest.mark.parametrize("M,N,K,bits", [(1, 7, 64, 8), (3, 5, 256, 8), (8, 8, 128, 8),
                                        (2, 6, 96, 4), (5, 3, 256, 4)])
def test_qgemm_vs_dequantized_matmul(M, N, K, bits):
    rng = np.random.default_rng(100 + M * N + K + bits)
    x = rng.standard_normal((M, K)).astype(np.float32)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    qx, dx = oracle.quantize_act_q8(x)
    if bits == 8:
        qw, dw = oracle.quantize_w_q8_0(w)
        qwv = qw
    else:
        qw, dw = oracle.quantize_w_q4_0(w)
        qwv = _unpack_q4(qw)
    y, mag = oracle.qgemm(qx, dx, qw, dw, bits)
    ref = _dequant_matmul(qx, dx, qwv, dw)
    # y is the binary64 sum rounded once to binary32
    assert np.all(np.abs(y - ref) <= 2.0 ** -24 * np.abs(ref) + 1e-12 * mag)
    # the dequantized values themselves approximate x @ w^T
    assert np.allclose(ref, x.astype(np.float64) @ w.astype(np.float64).T, rtol=0.05,
                       atol=0.05 * np.abs(x).max() * np.abs(w).max() * np.sqrt(K))


def test_qgemm_closed_form_constant():
    M, N, K = 2, 3, 128
    G = K // 32
    c, a = np.float32(0.3), np.float32(-1.7)
    w = np.full((N, K), c, np.float32)
    x = np.full((M, K), a, np.float32)
    qx, dx = oracle.quantize_act_q8(x)
    qw, dw = oracle.quantize_w_q8_0(w)
    assert np.all(qx == -127) and np.all(qw == 127)
    y, _ = oracle.qgemm(qx, dx, qw, dw, 8)
    d16 = np.float64(np.float32(c / np.float32(127)).astype(np.float16))
    dxv = np.float64(np.float32(abs(a) / np.float32(127)))
    want = np.float32(-G * 32 * 127 * 127 * d16 * dxv)
    assert np.all(y == want)


def test_qgemm_closed_form_one_hot():
    N, K, k0 = 9, 96, 45
    g0 = k0 // 32
    w = _weights(N=N, K=K)
    qw, dw = oracle.quantize_w_q8_0(w)
    for v in (np.float32(2.75), np.float32(-0.001)):
        x = np.zeros((1, K), np.float32)
        x[0, k0] = v
        qx, dx = oracle.quantize_act_q8(x)
        y, _ = oracle.qgemm(qx, dx, qw, dw, 8)
        d16 = dw[:, g0].view(np.float16).astype(np.float64)
        dxv = np.float64(np.float32(abs(v) / np.float32(127)))
        want = (d16 * dxv * 127 * np.sign(v) * qw[:, k0]).astype(np.float32)
        assert np.array_equal(y[0], want)


def test_qgemm_zero_and_pow2_scaling():
    x = _act_data(4, M=3, K=128)
    w = _weights(N=6, K=128)
    qw, dw = oracle.quantize_w_q8_0(w)
    qx, dx = oracle.quantize_act_q8(np.zeros_like(x))
    y0, _ = oracle.qgemm(qx, dx, qw, dw, 8)
    assert np.all(y0 == 0)
    qx, dx = oracle.quantize_act_q8(x)
    y1, _ = oracle.qgemm(qx, dx, qw, dw, 8)
    qx2, dx2 = oracle.quantize_act_q8(x * np.float32(8.0))
    y2, _ = oracle.qgemm(qx2, dx2, qw, dw, 8)
    assert np.array_equal(y2, y1 * np.float32(8.0))


def test_qgemm_rows_matches_full():
    rng = np.random.default_rng(21)
    x = rng.standard_normal((10, 64)).astype(np.float32)
    w = _weights(N=7, K=64)
    qx, dx = oracle.quantize_act_q8(x)
    qw, dw = oracle.quantize_w_q8_0(w)
    y, mag = oracle.qgemm(qx, dx, qw, dw, 8)
    rows = np.array([9, 0, 4, 4])
    yr, mr = oracle.qgemm_rows(qx, dx, rows, qw, dw, 8)
    assert np.array_equal(yr, y[rows]) and np.array_equal(mr, mag[rows])


# ---------------------------------------------------------------- MoE

def _moe_small(seed=31, E=6, T=11, topk=3, N=8, K=64):
    rng = np.random.default_rng(seed)
    w = (rng.standard_normal((E, N, K)) * 0.02).astype(np.float32)
    qw4 = np.empty((E, N, K // 2), np.uint8)
    dw = np.empty((E, N, K // 32), np.uint16)
    for e in range(E):
        qw4[e], dw[e] = oracle.quantize_w_q4_0(w[e])
    ids = np.stack([rng.choice(E, topk, replace=False) for _ in range(T)]).astype(np.int32)
    return rng, qw4, dw, ids


def test_moe_route_vs_numpy():
    _, _, _, ids = _moe_small()
    E = 6
    counts, offsets, perm, bad = oracle.moe_route(ids, E)
    flat = ids.ravel()
    assert bad == 0
    assert np.array_equal(counts, np.bincount(flat, minlength=E))
    assert np.array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
    assert np.array_equal(perm, np.argsort(flat, kind="stable"))


def test_moe_route_invalid_ids():
    ids = np.array([[0, 5], [7, 1], [-1, 0]], np.int32)
    counts, offsets, perm, bad = oracle.moe_route(ids, 6)
    assert bad == 2
    assert counts.tolist() == [2, 1, 0, 0, 0, 1]
    assert perm.tolist() == [0, 5, 3, 1]


def test_moe_single_expert_equals_dense():
    rng, qw4, dw, _ = _moe_small()
    T, K = 11, 64
    x = rng.standard_normal((T, K)).astype(np.float32)
    qx, dx = oracle.quantize_act_q8(x)
    ids = np.full((T, 1), 4, np.int32)
    y, _, bad = oracle.grouped_qgemm_moe(qx, dx, ids, 0, qw4, dw)
    yd, _ = oracle.qgemm(qx, dx, qw4[4], dw[4], 4)
    assert bad == 0 and np.array_equal(y, yd)


def test_moe_rows_per_pair_and_token_permutation():
    rng, qw4, dw, ids = _moe_small()
    T, topk, K = ids.shape[0], ids.shape[1], 64
    x = rng.standard_normal((T, K)).astype(np.float32)
    qx, dx = oracle.quantize_act_q8(x)
    y, _, _ = oracle.grouped_qgemm_moe(qx, dx, ids, 0, qw4, dw)
    # each pair row equals the dense product of its token with its expert
    for p in range(T * topk):
        t, e = p // topk, ids.ravel()[p]
        yd, _ = oracle.qgemm(qx[t:t + 1], dx[t:t + 1], qw4[e], dw[e], 4)
        assert np.array_equal(y[p], yd[0])
    # permuting tokens permutes the output rows
    pi = rng.permutation(T)
    y2, _, _ = oracle.grouped_qgemm_moe(qx[pi], dx[pi], ids[pi], 0, qw4, dw)
    assert np.array_equal(y2.reshape(T, topk, -1), y.reshape(T, topk, -1)[pi])
    # mode 1: one activation row per pair (repeat tokens) gives the same result
    qxp, dxp = np.repeat(qx, topk, axis=0), np.repeat(dx, topk, axis=0)
    y3, _, _ = oracle.grouped_qgemm_moe(qxp, dxp, ids, 1, qw4, dw)
    assert np.array_equal(y3, y)


def test_moe_unrouted_rows_are_zero():
    rng, qw4, dw, ids = _moe_small()
    ids = ids.copy()
    ids[2, 1] = 99
    ids[5, 0] = -3
    x = rng.standard_normal((ids.shape[0], 64)).astype(np.float32)
    qx, dx = oracle.quantize_act_q8(x)
    y, _, bad = oracle.grouped_qgemm_moe(qx, dx, ids, 0, qw4, dw)
    assert bad == 2
    assert np.all(y[2 * 3 + 1] == 0) and np.all(y[5 * 3 + 0] == 0)


# ---------------------------------------------------------------- MoE steps around the GEMM

def test_silu_mul_closed_forms():
    """silu(0) = 0; sigmoid(1) = e / (1 + e); silu(v) - silu(-v) = v; silu(v) -> v and
    silu(-v) -> 0 for large v; up scales h linearly."""
    g = np.array([0.0, 1.0, -1.0, 3.0, -3.0, 40.0, -40.0, 0.5], np.float32)
    up = np.ones_like(g)
    gu = np.concatenate([g, up])[None, :]
    h = oracle.silu_mul(gu, g.size)[0]
    assert h[0] == 0.0
    e = np.e
    assert abs(h[1] - e / (1.0 + e)) < 1e-15
    assert abs((h[1] - h[2]) - 1.0) < 1e-15                  # silu(1) - silu(-1) = 1
    assert abs((h[3] - h[4]) - 3.0) < 1e-14
    assert abs(h[5] - 40.0) < 1e-12 and 0.0 > h[6] > -1e-15
    gu2 = np.concatenate([g, np.full_like(g, -2.5)])[None, :]
    h2 = oracle.silu_mul(gu2, g.size)[0]
    assert np.allclose(h2, -2.5 * h, rtol=1e-15, atol=0.0)


def test_silu_mul_layout_gate_then_up():
    """Columns [0, F) are the gate and [F, 2F) the up half; extra columns are ignored."""
    rng = np.random.default_rng(41)
    P, F = 3, 64
    gu = rng.standard_normal((P, 2 * F + 5)).astype(np.float32)
    h = oracle.silu_mul(gu, F)
    g64, u64 = gu[:, :F].astype(np.float64), gu[:, F:2 * F].astype(np.float64)
    # sigmoid from tanh: 1 / (1 + e^-v) = (1 + tanh(v / 2)) / 2
    ref = g64 * (1.0 + np.tanh(g64 / 2.0)) / 2.0 * u64
    assert np.allclose(h, ref, rtol=1e-14, atol=1e-300)


def test_moe_combine_pins():
    """One-hot weights select a slot's row; rows equal and weights summing to one give the
    row; permuting slots together with their weights changes nothing; mag = sum |w y|."""
    rng = np.random.default_rng(43)
    T, topk, N = 5, 4, 24
    y = rng.standard_normal((T * topk, N)).astype(np.float32)
    w = np.zeros((T, topk), np.float32)
    w[np.arange(T), np.arange(T) % topk] = 1.0
    out, mag = oracle.moe_combine(y, w)
    for t in range(T):
        assert np.array_equal(out[t], y[t * topk + t % topk].astype(np.float64))
    assert np.array_equal(mag, np.abs(out))
    yc = np.repeat(rng.standard_normal((T, 1, N)), topk, axis=1).reshape(T * topk, N).astype(np.float32)
    wq = np.full((T, topk), 0.25, np.float32)
    out_c, _ = oracle.moe_combine(yc, wq)
    assert np.allclose(out_c, yc[::topk].astype(np.float64), rtol=1e-15, atol=0)
    wr = rng.random((T, topk)).astype(np.float32)
    perm = rng.permutation(topk)
    out1, mag1 = oracle.moe_combine(y, wr)
    y_p = y.reshape(T, topk, N)[:, perm].reshape(T * topk, N)
    out2, mag2 = oracle.moe_combine(y_p, wr[:, perm])
    assert np.allclose(out1, out2, rtol=1e-14, atol=1e-14)
    assert np.allclose(mag1, mag2, rtol=1e-14, atol=0)
    assert np.allclose(mag1, np.abs(wr[:, :, None].astype(np.float64) *
                                    y.reshape(T, topk, N).astype(np.float64)).sum(1), rtol=1e-14)


# ---------------------------------------------------------------- GGUF block import

def _golden_gguf():
    vals = {}
    for line in open(os.path.join(GOLD, "gguf_blocks.txt")):
        if line.startswith("#") or not line.strip():
            continue
        key, *rest = line.split()
        vals[key] = rest
    return vals


def test_gguf_import_golden_blocks():
    g = _golden_gguf()
    q8 = np.array([int(b, 16) for b in g["q8_bytes"]], np.uint8)
    q, d = oracle.import_gguf(q8, 1, 32, 8)
    assert d[0, 0] == int(g["q8_scale"][0], 16)
    assert np.array_equal(q[0], np.array([int(v) for v in g["q8_values"]], np.int8))
    q4 = np.array([int(b, 16) for b in g["q4_bytes"]], np.uint8)
    q4c, d4 = oracle.import_gguf(q4, 1, 32, 4)
    assert d4[0, 0] == int(g["q4_scale"][0], 16)
    # unpack the planar nibbles with the header's rule (byte j: element j low, j+16 high)
    b = [int(v) for v in q4c[0]]
    vals = [(b[j] & 15) - 8 for j in range(16)] + [(b[j] >> 4) - 8 for j in range(16)]
    assert vals == [int(v) for v in g["q4_values"]]


def _encode_gguf(q, d, wbits):
    """Independent writer of the GGUF block layout with struct (little-endian)."""
    import struct
    N, G = d.shape
    cb = 32 if wbits == 8 else 16
    out = bytearray()
    for n in range(N):
        for g in range(G):
            out += struct.pack("<H", int(d[n, g]))
            out += q[n, g * cb:(g + 1) * cb].astype(np.uint8).tobytes()
    return np.frombuffer(bytes(out), np.uint8)


@pytest.mark.parametrize("wbits", [8, 4])
def test_gguf_import_round_trip(wbits):
    """Quantize planar, write GGUF blocks independently, import: the planes come back."""
    rng = np.random.default_rng(5 + wbits)
    N, K = 7, 256
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    q, d = oracle.quantize_w_q8_0(w) if wbits == 8 else oracle.quantize_w_q4_0(w)
    blocks = _encode_gguf(q, d, wbits)
    assert blocks.size == N * (K // 32) * (34 if wbits == 8 else 18)
    q2, d2 = oracle.import_gguf(blocks, N, K, wbits)
    assert np.array_equal(q2.view(np.uint8), q.view(np.uint8)) and np.array_equal(d2, d)


# ---------------------------------------------------------------- split-K attention merge

def _partials(scores, values, bounds):
    """Per-split partials from the definition of softmax attention (numpy, binary64)."""
    S = len(bounds) - 1
    R, T = scores.shape
    D = values.shape[2]
    m = np.full((S, R), -np.inf)
    l = np.zeros((S, R))
    acc = np.zeros((S, R, D))
    for s in range(S):
        a, b = bounds[s], bounds[s + 1]
        if a == b:
            continue
        x = scores[:, a:b]
        m[s] = x.max(axis=1)
        e = np.exp(x - m[s][:, None])
        l[s] = e.sum(axis=1)
        acc[s] = np.einsum("rt,rtd->rd", e, values[:, a:b])
    return m, l, acc


def test_splitk_merge_equals_unsplit_softmax():
    """Merging the splits of a row gives softmax(scores) @ values and log-sum-exp of the
    scores, however the keys are split (including empty splits)."""
    rng = np.random.default_rng(77)
    R, T, D = 6, 50, 16
    scores = rng.standard_normal((R, T)) * 3.0
    values = rng.standard_normal((R, T, D))
    p = np.exp(scores - scores.max(axis=1, keepdims=True))
    ref = np.einsum("rt,rtd->rd", p / p.sum(axis=1, keepdims=True), values)
    ref_lse = np.log(np.exp(scores).sum(axis=1))
    for bounds in ([0, T], [0, 10, 10, 33, T], list(range(0, T + 1, 5))):
        m, l, acc = _partials(scores, values, bounds)
        out, lse, mag = oracle.splitk_merge(m.astype(np.float32), l.astype(np.float32),
                                            acc.astype(np.float32))
        assert np.allclose(out, ref, rtol=1e-5, atol=1e-6)     # binary32 partials in
        assert np.allclose(lse, ref_lse, rtol=1e-6, atol=1e-6)
        assert np.all(mag >= np.abs(out) - 1e-12)


def test_splitk_merge_single_split_and_empty_rows():
    rng = np.random.default_rng(78)
    acc = rng.standard_normal((1, 3, 8)).astype(np.float32)
    m = np.array([[0.5, -2.0, 3.0]], np.float32)
    l = np.array([[2.0, 4.0, 0.5]], np.float32)
    out, lse, _ = oracle.splitk_merge(m, l, acc)
    assert np.allclose(out, acc[0] / l[0][:, None], rtol=1e-15)
    assert np.allclose(lse, m[0] + np.log(l[0]), rtol=1e-15)
    me = np.full((3, 2), -np.inf, np.float32)
    me[1, 0] = 1.0
    le = np.zeros((3, 2), np.float32)
    le[1, 0] = 3.0
    acce = np.zeros((3, 2, 4), np.float32)
    acce[1, 0] = [3.0, 6.0, -3.0, 0.0]
    out, lse, _ = oracle.splitk_merge(me, le, acce)
    assert np.array_equal(out[0], [1.0, 2.0, -1.0, 0.0]) and np.isclose(lse[0], 1.0 + np.log(3.0))
    assert np.array_equal(out[1], np.zeros(4)) and lse[1] == -np.inf


# ---------------------------------------------------------------- 3-bit WHT + Lloyd-Max KV codec

@pytest.mark.parametrize("D", [64, 128, 256])
def test_wht_matches_sylvester_hadamard(D):
    """The transform is scipy's Sylvester Hadamard matrix over sqrt(D), orthonormal and its
    own inverse."""
    sl = pytest.importorskip("scipy.linalg")
    rng = np.random.default_rng(D)
    x = rng.standard_normal((5, D))
    H = sl.hadamard(D) / np.sqrt(D)
    y = oracle.wht(x)
    assert np.allclose(y, x @ H.T, rtol=1e-12, atol=1e-12)
    assert np.allclose(oracle.wht(y), x, rtol=1e-12, atol=1e-12)
    assert np.allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)


def test_lloyd_max_codebook_conditions():
    """Each level is the mean of N(0,1) over its cell and each threshold the midpoint of its
    two levels (checked by numerical quadrature, not by the oracle's closed form); the
    codebook is symmetric and its mean squared error is a local minimum."""
    integ = pytest.importorskip("scipy.integrate")
    lv, th = oracle.kv3_codebook()
    assert np.all(np.diff(lv) > 0) and np.allclose(lv, -lv[::-1], atol=1e-15)
    assert np.allclose(th, (lv[:-1] + lv[1:]) / 2, rtol=0, atol=1e-15)
    phi = lambda t: np.exp(-t * t / 2) / np.sqrt(2 * np.pi)
    edges = np.concatenate([[-np.inf], th, [np.inf]])
    for k in range(8):
        mass = integ.quad(phi, edges[k], edges[k + 1])[0]
        mean = integ.quad(lambda t: t * phi(t), edges[k], edges[k + 1])[0] / mass
        assert abs(mean - lv[k]) < 1e-9

    def mse(levels):
        e = np.concatenate([[-np.inf], (levels[:-1] + levels[1:]) / 2, [np.inf]])
        return sum(integ.quad(lambda t: (t - levels[k]) ** 2 * phi(t), e[k], e[k + 1])[0]
                   for k in range(8))

    base = mse(lv)
    assert 0.0344 < base < 0.0347                    # 3-bit Gaussian Lloyd-Max distortion
    for k in (0, 3, 6):
        for dlt in (1e-3, -1e-3):
            p = lv.copy()
            p[k] += dlt
            assert mse(p) > base


def _unpack_kv3(codes, D):
    E = D // 32
    T = codes.shape[0]
    k = np.zeros((T, D), np.int64)
    for j in range(D):
        L, e = divmod(j, E)
        for b in range(3):
            k[:, j] |= ((codes[:, b * E + e].astype(np.int64) >> L) & 1) << b
    return k


@pytest.mark.parametrize("D", [64, 128, 256])
def test_kv3_hadamard_column_closed_form(D):
    """x = a Hadamard column: y = sqrt(D) e_k, s = 1, the code of y_k is 7 and every other
    code is 4 (u = 0 sits on the middle threshold); decoding gives H (l_7 e_k + l_4 (1 - e_k))."""
    sl = pytest.importorskip("scipy.linalg")
    H = sl.hadamard(D).astype(np.float64)
    k = 5
    x = H[:, k].astype(np.float32)[None, :]
    codes, scales, _ = oracle.kv3_encode(x)
    assert scales[0] == 1.0
    c = _unpack_kv3(codes, D)[0]
    assert c[k] == 7 and np.all(np.delete(c, k) == 4)
    lv, _ = oracle.kv3_codebook()
    lv32 = lv.astype(np.float32).astype(np.float64)
    yhat = np.full(D, lv32[4])
    yhat[k] = lv32[7]
    assert np.allclose(oracle.kv3_decode(codes, scales, D)[0], H @ yhat / np.sqrt(D), rtol=1e-12)


def test_kv3_gaussian_distortion_and_zero_vector():
    """On Gaussian vectors the relative error of decode(encode(x)) is the Lloyd-Max
    distortion; a zero vector codes to scale 0 and decodes to 0."""
    rng = np.random.default_rng(13)
    D = 128
    x = rng.standard_normal((4000, D)).astype(np.float32)
    x[0] = 0.0
    codes, scales, _ = oracle.kv3_encode(x)
    xr = oracle.kv3_decode(codes, scales, D)
    assert scales[0] == 0.0 and np.all(xr[0] == 0.0)
    rel = np.sum((xr[1:] - x[1:]) ** 2) / np.sum(x[1:].astype(np.float64) ** 2)
    assert 0.030 < rel < 0.040
