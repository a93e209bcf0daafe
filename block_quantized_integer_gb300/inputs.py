"""Seeded synthetic workloads for the block-quantized integer GEMM/GEMV.

This module only draws random numbers.  It holds none of the method's
arithmetic (no quantization, no dot products, no scaling), so both the CPU
oracle and the CUDA path can take their inputs from it without sharing any
computation.

The value distributions follow the workloads of the pages this library is
built from: Q8_0 projections of a dense LLM layer (weights ~ N(0, 0.02),
activations ~ N(0, 1) with a few outlier entries or outlier channels), and a
128-expert MoE layer with 947 prompt tokens routed top-8 by a Zipf-skewed
expert popularity ("A 35B Hybrid-Attention Mixture-of-Experts Model on a 6GB
2011 GPU", Methodology 1 and 2, Results).

Generator: NumPy ``default_rng`` (PCG64).  Seed = ``BASE_SEED + workload
index``; within one workload the draw order is weights, activations, outlier
selection, routing.
"""
from __future__ import annotations

import numpy as np

BASE_SEED = 20261202

# Workload indices (the seed offset of each).
PARITY = 0      # Q8_0 W8A8 M=4 N=256 K=512, everything ~ N(0, 1)
DECODE = 1      # M=1 / M=4 GEMV over four projection shapes
PREFILL = 2     # M=2048 GEMM, two shapes
MOE = 3         # grouped W4A8, 128 experts, 947 tokens, top-8 Zipf(1.1)
LONGCTX = 4     # M=18432 GEMM, two shapes

DECODE_SHAPES = ((4096, 4096), (12288, 4096), (4096, 12288), (151936, 4096))  # (N, K)
PREFILL_SHAPES = ((2048, 12288, 4096), (2048, 4096, 12288))                   # (M, N, K)
LONGCTX_SHAPES = ((18432, 17408, 5120), (18432, 5120, 17408))                 # (M, N, K)
MOE_EXPERTS = 128
MOE_TOKENS = 947
MOE_TOPK = 8
MOE_GATE_UP = (2048, 2048)   # (N, K): gate rows 0..1023 then up rows 1024..2047
MOE_DOWN = (2048, 1024)      # (N, K)
MOE_ZIPF_S = 1.1


def rng_for(workload: int, sub: int = 0) -> np.random.Generator:
    """PCG64 generator for one workload (``sub`` separates independent shapes)."""
    return np.random.default_rng([BASE_SEED + workload, sub])


def normal(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    a = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return a


def with_entry_outliers(rng, x: np.ndarray, frac: float, factor: float) -> np.ndarray:
    """Scale round(frac*K) entries of every row (chosen per row, no replacement)."""
    M, K = x.shape
    n_out = int(round(frac * K))
    for m in range(M):
        idx = rng.choice(K, size=n_out, replace=False)
        x[m, idx] *= np.float32(factor)
    return x


def with_channel_outliers(rng, x: np.ndarray, frac: float, factor: float) -> np.ndarray:
    """Scale round(frac*K) columns of x, the same columns in every row."""
    K = x.shape[1]
    n_out = int(round(frac * K))
    idx = rng.choice(K, size=n_out, replace=False)
    x[:, idx] *= np.float32(factor)
    return x


def parity_case(M: int = 4, N: int = 256, K: int = 512, sub: int = 0):
    """Weights [N,K] and activations [M,K], both ~ N(0, 1)."""
    rng = rng_for(PARITY, sub)
    w = normal(rng, (N, K))
    x = normal(rng, (M, K))
    return w, x


def decode_case(N: int, K: int, M: int = 1, sub: int = 0):
    """Weights ~ N(0, 0.02); activations ~ N(0, 1) with 1% of each row x20."""
    rng = rng_for(DECODE, sub)
    w = normal(rng, (N, K), 0.02)
    x = normal(rng, (M, K))
    with_entry_outliers(rng, x, 0.01, 20.0)
    return w, x


def prefill_case(M: int, N: int, K: int, sub: int = 0, channel_frac: float = 0.005,
                 factor: float = 30.0, workload: int = PREFILL):
    """Weights ~ N(0, 0.02); activations ~ N(0, 1) with outlier K-columns."""
    rng = rng_for(workload, sub)
    w = normal(rng, (N, K), 0.02)
    x = normal(rng, (M, K))
    with_channel_outliers(rng, x, channel_frac, factor)
    return w, x


def longctx_case(M: int, N: int, K: int, sub: int = 0):
    """Like the prefill case with 1% of K-columns x20."""
    return prefill_case(M, N, K, sub=sub, channel_frac=0.01, factor=20.0, workload=LONGCTX)


def zipf_routing(rng, T: int, E: int, topk: int, s: float = MOE_ZIPF_S) -> np.ndarray:
    """topk distinct experts per token; expert e drawn with p(e) ~ (1 + pi(e))^-s,
    pi a seeded permutation of the experts.  Returns int32 [T, topk]."""
    perm = rng.permutation(E)
    p = (1.0 + perm.astype(np.float64)) ** (-s)
    p /= p.sum()
    ids = np.empty((T, topk), dtype=np.int32)
    for t in range(T):
        ids[t] = rng.choice(E, size=topk, replace=False, p=p)
    return ids


def moe_case(E: int = MOE_EXPERTS, T: int = MOE_TOKENS, topk: int = MOE_TOPK,
             gate_up=MOE_GATE_UP, down=MOE_DOWN, sub: int = 0):
    """Expert weights, token activations and routing of the MoE workload.

    Returns dict with w_gate_up [E,N1,K1], w_down [E,N2,K2] (fp32), x_tok [T,K1],
    x_pair [T*topk,K2] (fp32), topk_ids [T,topk] int32 and route_w [T,topk] fp32
    (router weights of each token's slots, positive, summing to one; drawn last so
    the other arrays do not depend on them)."""
    rng = rng_for(MOE, sub)
    N1, K1 = gate_up
    N2, K2 = down
    w1 = normal(rng, (E, N1, K1), 0.02)
    w2 = normal(rng, (E, N2, K2), 0.02)
    x_tok = normal(rng, (T, K1))
    x_pair = normal(rng, (T * topk, K2))
    ids = zipf_routing(rng, T, E, topk)
    rw = rng.random((T, topk)) + 0.05
    rw = (rw / rw.sum(axis=1, keepdims=True)).astype(np.float32)
    return dict(w_gate_up=w1, w_down=w2, x_tok=x_tok, x_pair=x_pair, topk_ids=ids, route_w=rw)
