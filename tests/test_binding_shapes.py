"""The Python binding rejects mis-shaped outputs and operands before anything
reaches the library (a short y would otherwise be written past its end by the
kernels).  Shapes are checked before devices, so CPU tensors exercise the
checks here without a GPU; no call reaches a launch."""
import pytest
import torch

import block_quantized_integer_gb300 as qg


def _moe(T=5, topk=2, E=3, N=16, K=64, rows_x=None):
    rows_x = T if rows_x is None else rows_x
    return dict(qx=torch.zeros((rows_x, K), dtype=torch.int8),
                dx=torch.zeros((rows_x, K // 32), dtype=torch.float32),
                topk_ids=torch.zeros((T, topk), dtype=torch.int32),
                qw4=torch.zeros((E, N, K // 2), dtype=torch.uint8),
                dw=torch.zeros((E, N, K // 32), dtype=torch.float16))


@pytest.mark.parametrize("fn", [qg.grouped_qgemm_moe, qg.grouped_qgemm_moe_noalloc])
def test_moe_short_y_rejected(fn):
    a = _moe()
    y = torch.zeros((5 * 2 - 1, 16), dtype=torch.float32)           # one row short
    err = torch.zeros(1, dtype=torch.int32)
    with pytest.raises(ValueError, match="y must be"):
        fn(a["qx"], a["dx"], a["topk_ids"], 0, a["qw4"], a["dw"], y, err)
    y = torch.zeros((10, 15), dtype=torch.float32)                    # one column short
    with pytest.raises(ValueError, match="y must be"):
        fn(a["qx"], a["dx"], a["topk_ids"], 0, a["qw4"], a["dw"], y, err)


@pytest.mark.parametrize("fn", [qg.grouped_qgemm_moe, qg.grouped_qgemm_moe_noalloc])
def test_moe_operand_shapes_rejected(fn):
    a = _moe()
    y = torch.zeros((10, 16), dtype=torch.float32)
    err = torch.zeros(1, dtype=torch.int32)
    bad = dict(a)
    bad["qw4"] = torch.zeros((3, 16, 31), dtype=torch.uint8)         # K/2 - 1 bytes a row
    with pytest.raises(ValueError, match="qw4"):
        fn(bad["qx"], bad["dx"], bad["topk_ids"], 0, bad["qw4"], bad["dw"], y, err)
    bad = dict(a)
    bad["dw"] = torch.zeros((3, 15, 2), dtype=torch.float16)          # a scale row short
    with pytest.raises(ValueError, match="dw"):
        fn(bad["qx"], bad["dx"], bad["topk_ids"], 0, bad["qw4"], bad["dw"], y, err)
    bad = dict(a)
    bad["dx"] = torch.zeros((4, 2), dtype=torch.float32)              # an activation row short
    with pytest.raises(ValueError, match="dx"):
        fn(bad["qx"], bad["dx"], bad["topk_ids"], 0, bad["qw4"], bad["dw"], y, err)
    with pytest.raises(ValueError, match="d_err"):
        fn(a["qx"], a["dx"], a["topk_ids"], 0, a["qw4"], a["dw"], y,
           torch.zeros(0, dtype=torch.int32))


def test_noalloc_needs_outputs():
    a = _moe()
    with pytest.raises(ValueError, match="allocates nothing"):
        qg.grouped_qgemm_moe_noalloc(a["qx"], a["dx"], a["topk_ids"], 0, a["qw4"], a["dw"],
                                     None, None)


@pytest.mark.parametrize("fn,wdt,kfac", [(qg.qgemm_q8_0, torch.int8, 1),
                                         (qg.qgemm_q4_0, torch.uint8, 2)])
def test_dense_short_y_rejected(fn, wdt, kfac):
    M, N, K = 9, 40, 256
    qx = torch.zeros((M, K), dtype=torch.int8)
    dx = torch.zeros((M, K // 32), dtype=torch.float32)
    qw = torch.zeros((N, K // kfac), dtype=wdt)
    dw = torch.zeros((N, K // 32), dtype=torch.float16)
    for shape in ((M - 1, N), (M, N - 1)):
        with pytest.raises(ValueError, match="y must have at least"):
            fn(qx, dx, qw, dw, y=torch.zeros(shape, dtype=torch.float32))
    # a wider, strided view is a valid y
    with pytest.raises(ValueError, match="CUDA tensor"):
        fn(qx, dx, qw, dw, y=torch.zeros((M, 2 * N), dtype=torch.float32)[:, :N])
