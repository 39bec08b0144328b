"""GPU parity on the seeded workloads at their full sizes, through the C ABI,
against the CPU oracle: every element of every output, except on the
BatchNorm workloads of the page's (64, 64, 112, 112) shape, where the GPU runs
the full tensor and every element of three channels (first, middle, last) is
checked against the oracle run on those channels alone (BatchNorm channels
are independent).

With NRM_PARITY_REPORT set to a file name, each workload appends one JSON line
with its measured errors: the largest error, the largest ulp distance and how
many 16-bit elements passed on the cancellation bound rather than within 1 ulp
(n_cancel_floor)."""
import json
import os

import pytest
import torch

import runners as RN
from row_wise_normalization_reduce_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import row_wise_normalization_reduce_gb300 as nrm
    nrm.build()
    nrm.force_plan(nrm.PLAN_AUTO)
    yield


SAMPLED = 20_000_000  # elements above which BatchNorm channels are sampled


@pytest.mark.parametrize("w", W.ALL, ids=lambda w: w.name)
def test_workload_full_size(orc, w):
    inp = W.make_inputs(w)
    gpu = RN.run_gpu(w.op, inp, w.eps, w.momentum)
    if w.op.startswith("bn") and inp["x"].numel() > SAMPLED:
        c = inp["x"].shape[1]
        chans = [0, c // 2, c - 1]
        inp = RN.select_channels(w.op, inp, chans)
        gpu = RN.slice_gpu_channels(gpu, chans)
    ref = RN.run_oracle(orc, w.op, inp, w.eps, w.momentum)
    rep = RN.compare(w.op, inp, gpu, ref)
    print(w.name, rep)
    path = os.environ.get("NRM_PARITY_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"workload": w.name, "checked_elements": int(inp["x"].numel()),
                                "errors": rep}, default=float) + "\n")


def test_add_rms_inplace_residual(orc):
    w = W.ADD_RMS_BF16_4096x4096
    inp = W.make_inputs(w, shape=(512, 4096))
    gpu = RN.run_gpu(w.op, inp, w.eps, residual_inplace=True)
    ref = RN.run_oracle(orc, w.op, inp, w.eps)
    RN.compare(w.op, inp, gpu, ref)


@pytest.mark.parametrize("w", [W.ADD_RMS_BF16_4096x4096, W.LN_BF16_4096x4096,
                               W.BN_F32_32x64x56x56], ids=lambda w: w.name)
def test_repeatable_bitwise(w):
    inp = W.make_inputs(w)
    a = RN.run_gpu(w.op, inp, w.eps, w.momentum)
    b = RN.run_gpu(w.op, inp, w.eps, w.momentum)
    for k in a:
        assert (a[k] == b[k]).all(), k


def test_on_non_default_stream(orc):
    import row_wise_normalization_reduce_gb300 as nrm
    w = W.LN_F32_64x1024
    inp = W.make_inputs(w)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        x = inp["x"].cuda()
        g = inp["gamma"].cuda()
        b = inp["beta"].cuda()
        y, mean, rstd = nrm.ln_fwd(x, g, b, w.eps)
    s.synchronize()
    ref = RN.run_oracle(orc, "ln", inp, w.eps)
    RN.compare("ln", inp, {"y": RN.B.torch_to_np(y.cpu()), "mean": mean.cpu().numpy(),
                           "rstd": rstd.cpu().numpy()}, ref)
