"""The decode stand-in GEMV against a CPU fp64 GEMV of the same bf16 inputs.

Tolerance: fp32 products of bf16 values are exact; summing 2,560 of them in
fp32 (fma chain per lane, then a 32-way tree) loses at most about
(terms x 2^-24) of sum |W_rc x_c| per row, so |y - y_ref| <= 1e-4 * sum |W x|
leaves a wide margin.
"""

import numpy as np
import pytest
import torch

from expert_host_block_gb300 import kvx

pytestmark = pytest.mark.gpu


def _ref(W16, x16):
    W = W16.float().cpu().numpy().astype(np.float64)
    x = x16.float().cpu().numpy().astype(np.float64)
    return W @ x, np.abs(W) @ np.abs(x)


@pytest.mark.parametrize("rows,cols,ctas", [(4096, 2560, 0), (1000, 256, 3), (777, 4096, 0), (5, 2560, 152)])
def test_gemv_matches_fp64(rows, cols, ctas):
    g = torch.Generator(device="cuda").manual_seed(rows * 7 + cols)
    W = (torch.rand(rows, cols, device="cuda", generator=g) * 2 - 1).to(torch.bfloat16)
    x = (torch.rand(cols, device="cuda", generator=g) * 2 - 1).to(torch.bfloat16)
    y = torch.full((rows,), float("nan"), device="cuda", dtype=torch.float32)
    kvx.kvx_standin_gemv_bf16(W.data_ptr(), x.data_ptr(), y.data_ptr(), rows, cols, ctas,
                              torch.cuda.current_stream())
    torch.cuda.synchronize()
    want, mag = _ref(W, x)
    got = y.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - want) <= 1e-4 * mag + 1e-6)


def test_gemv_rejects_bad_shapes():
    W = torch.zeros(16, 512, device="cuda", dtype=torch.bfloat16)
    x = torch.zeros(512, device="cuda", dtype=torch.bfloat16)
    y = torch.zeros(16, device="cuda", dtype=torch.float32)
    for cols in (100, 8192):
        with pytest.raises(kvx.KvxError):
            kvx.kvx_standin_gemv_bf16(W.data_ptr(), x.data_ptr(), y.data_ptr(), 16, cols)
    with pytest.raises(kvx.KvxError):
        kvx.kvx_standin_gemv_bf16(W.data_ptr() + 2, x.data_ptr(), y.data_ptr(), 16, 512)
