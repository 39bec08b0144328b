"""Strided rows (the *_ld entry points) on the GPU: inputs and outputs as
column slices of padded buffers, with row strides that keep 16-byte row
starts (vector kernels) and strides that do not (scalar kernel); y written
into other columns of the input's own buffer; the padding must stay
untouched.  Compared with the oracle on contiguous copies."""
import numpy as np
import pytest
import torch

import runners as RN
import row_wise_normalization_reduce_gb300 as nrm
from row_wise_normalization_reduce_gb300 import workloads as W

pytestmark = pytest.mark.gpu

POISON = -7.25


@pytest.fixture(scope="module", autouse=True)
def _lib():
    nrm.build()
    nrm.force_plan(nrm.PLAN_AUTO)
    yield


def _padded(t, ld, col0=0, width=None):
    """A [rows, ld] device buffer filled with POISON and t copied into columns
    [col0, col0 + N); returns (buffer, view)."""
    rows, n = t.shape
    buf = torch.full((rows, ld), POISON, dtype=t.dtype, device="cuda")
    view = buf[:, col0:col0 + n]
    view.copy_(t.cuda())
    return buf, view


@pytest.mark.parametrize("op", ["ln", "rms", "add_rms", "softmax"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("n,pad", [(1024, 4), (1024, 8), (1024, 16), (4096, 8), (1000, 3),
                                   (64, 64), (16384, 8)])
def test_strided_rows(orc, op, dtype, n, pad):
    rows = 24 if n <= 4096 else 4
    inp = W.generic_rows(op, dtype, rows, n, seed=n + pad)
    ld = n + pad
    xbuf, x = _padded(inp["x"], ld)
    ybuf = torch.full((rows, ld), POISON, dtype=x.dtype, device="cuda")
    y = ybuf[:, pad:pad + n] if pad >= 1 else ybuf[:, :n]
    d = {k: v.cuda() for k, v in inp.items() if k not in ("x", "residual")}
    if op == "ln":
        nrm.ln_fwd(x, d["gamma"], d["beta"], 1e-5, out=y)
    elif op == "rms":
        nrm.rms_fwd(x, d["w"], 1e-6, out=y)
    elif op == "softmax":
        nrm.softmax_fwd(x, out=y)
    else:
        rbuf, r = _padded(inp["residual"], ld + 8)
        robuf = torch.full((rows, ld * 2), POISON, dtype=x.dtype, device="cuda")
        ro = robuf[:, ld:ld + n]
        nrm.add_rms_fwd(x, r, d["w"], 1e-6, residual_out=ro, out=y)
    torch.cuda.synchronize()
    eps = 1e-5 if op == "ln" else 1e-6
    ref = RN.run_oracle(orc, op, inp, eps)
    gpu = {"y": RN.B.torch_to_np(y.contiguous().cpu())}
    dt = RN.B.dt_code(x.dtype)
    if op == "softmax":
        RN.T.check_softmax(dt, gpu["y"], ref["y"], ref["y_wide"])
    elif op == "ln":
        scale = RN.T.ln_affine_scale(dt, RN.to_np(inp)["x"], ref["mean"], ref["rstd"],
                                     RN.to_np(inp)["gamma"], RN.to_np(inp)["beta"])
        RN.T.check_y(dt, gpu["y"], ref["y"], ref["y_wide"], scale)
    else:
        RN.T.check_y(dt, gpu["y"], ref["y"], ref["y_wide"], None)
    if op == "add_rms":
        assert np.array_equal(RN.B.torch_to_np(ro.contiguous().cpu()), ref["residual_out"])
        assert torch.all(robuf[:, :ld] == POISON) and torch.all(robuf[:, ld + n:] == POISON)
    # padding untouched, input untouched
    assert torch.all(ybuf[:, :pad] == POISON) and torch.all(ybuf[:, pad + n:] == POISON)
    assert torch.all(xbuf[:, n:] == POISON)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_output_in_other_columns_of_input_buffer(orc, dtype):
    # y shares one padded buffer with x: x in columns [0, N), y in [N, 2N)
    rows, n = 16, 2048
    inp = W.generic_rows("ln", dtype, rows, n, seed=9)
    buf = torch.full((rows, 2 * n + 8), POISON, dtype=W.DTYPES[dtype], device="cuda")
    x = buf[:, :n]
    x.copy_(inp["x"].cuda())
    y = buf[:, n:2 * n]
    nrm.ln_fwd(x, inp["gamma"].cuda(), inp["beta"].cuda(), 1e-5, out=y)
    torch.cuda.synchronize()
    ref = RN.run_oracle(orc, "ln", inp, 1e-5)
    dt = RN.B.dt_code(x.dtype)
    n_ = RN.to_np(inp)
    scale = RN.T.ln_affine_scale(dt, n_["x"], ref["mean"], ref["rstd"], n_["gamma"], n_["beta"])
    RN.T.check_y(dt, RN.B.torch_to_np(y.contiguous().cpu()), ref["y"], ref["y_wide"], scale)
    assert np.array_equal(RN.B.torch_to_np(x.contiguous().cpu()), n_["x"])
    assert torch.all(buf[:, 2 * n:] == POISON)


def test_strided_plans_match_contiguous():
    # every forced plan gives the same bits on a strided view as on a copy
    inp = W.generic_rows("rms", "bf16", 64, 4096, seed=4)
    xbuf, x = _padded(inp["x"], 4096 + 64)
    xc = inp["x"].cuda()
    w = inp["w"].cuda()
    for plan in ([nrm.PLAN_AUTO], [nrm.PLAN_CTA, 256, 2], [nrm.PLAN_PERSIST, 256, 2],
                 [nrm.PLAN_TMA, 128, 4, 2, 2], [nrm.PLAN_GENERIC, 256], [nrm.PLAN_WRAW, 256, 16]):
        nrm.force_plan(*plan)
        a, _ = nrm.rms_fwd(x, w, 1e-6)
        b, _ = nrm.rms_fwd(xc, w, 1e-6)
        torch.cuda.synchronize()
        assert torch.equal(a, b), plan
    nrm.force_plan(nrm.PLAN_AUTO)
