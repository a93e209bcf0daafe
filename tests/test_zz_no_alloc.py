"""grouped_qgemm_moe_noalloc: the MoE GEMM entry point that allocates nothing.

It exists for callers that cannot allocate device memory (a serving process
whose memory is reserved up front by its own pool, a plugin host that grants
no allocation rights): the routing scratch lives in a fixed array inside the
library.  Its output must match the oracle's y, and the workspace-taking
grouped_qgemm_moe's, within the tolerance of the other parity tests, on two
calls in a row (the second call reuses the array the first one left behind).
Collected last on purpose.
"""
import numpy as np
import pytest
import torch

import oracle
import block_quantized_integer_gb300 as qg
from block_quantized_integer_gb300 import inputs
from helpers import RTOL, assert_close, dev, to_dev, to_np

pytestmark = pytest.mark.gpu


def _case(seed, E=12, T=97, topk=4, N=160, K=256):
    rng = np.random.default_rng(seed)
    w = (rng.standard_normal((E, N, K)) * 0.02).astype(np.float32)
    qw4 = np.empty((E, N, K // 2), np.uint8)
    dw = np.empty((E, N, K // 32), np.uint16)
    for e in range(E):
        qw4[e], dw[e] = oracle.quantize_w_q4_0(w[e])
    ids = inputs.zipf_routing(rng, T, E, topk)
    x = rng.standard_normal((T, K)).astype(np.float32)
    qx, dx = oracle.quantize_act_q8(x)
    return qx, dx, ids, qw4, dw


def test_noalloc_matches_workspace_entry_twice():
    # two different problems back to back, so the second call sees the first
    # call's leftovers in the shared scratch array
    for seed, (T, topk) in ((1, (97, 4)), (2, (53, 8))):
        qx, dx, ids, qw4, dw = _case(seed, T=T, topk=topk)
        args = (to_dev(qx), to_dev(dx), to_dev(ids), 0, to_dev(qw4), to_dev(dw))
        y_ref, err_ref = qg.grouped_qgemm_moe(*args)
        y = torch.full_like(y_ref, 3.0)
        d_err = torch.zeros(1, dtype=torch.int32, device=dev())
        qg.grouped_qgemm_moe_noalloc(*args, y, d_err)
        torch.cuda.synchronize()
        assert int(d_err.item()) == 0 and int(err_ref.item()) == 0
        y_oracle, mag, _ = oracle.grouped_qgemm_moe(qx, dx, ids, 0, qw4, dw)
        assert_close(to_np(y), y_oracle, mag)
        # and the workspace entry point: a different kernel, each within the bar of the
        # oracle, so the two within twice that bar of each other
        assert_close(to_np(y), to_np(y_ref), mag, rtol=2 * RTOL)


def test_noalloc_rejects_oversize_before_launch():
    qx = torch.zeros((70000, 64), dtype=torch.int8, device=dev())
    dx = torch.zeros((70000, 2), dtype=torch.float32, device=dev())
    ids = torch.zeros((70000, 1), dtype=torch.int32, device=dev())
    qw4 = torch.zeros((2, 16, 32), dtype=torch.uint8, device=dev())
    dw = torch.zeros((2, 16, 2), dtype=torch.float16, device=dev())
    y = torch.zeros((70000, 16), dtype=torch.float32, device=dev())
    d_err = torch.zeros(1, dtype=torch.int32, device=dev())
    with pytest.raises(qg.QGError) as ei:
        qg.grouped_qgemm_moe_noalloc(qx, dx, ids, 0, qw4, dw, y, d_err)
    assert ei.value.name == "QG_ERR_UNSUPPORTED"
