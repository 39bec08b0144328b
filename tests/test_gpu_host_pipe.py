"""add_rms_fwd_host: the fused residual add + RMSNorm on host tensors,
streamed through the device in chunks.  Outputs against the oracle (residual_out
bit-exact), for row counts that leave a ragged last chunk, fewer rows than one
chunk, several dtypes, page-locked and ordinary host memory, and the residual
stream updated in place on the host."""
import numpy as np
import pytest
import torch

import runners as RN
import row_wise_normalization_reduce_gb300 as nrm
from row_wise_normalization_reduce_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    nrm.build()
    nrm.force_plan(nrm.PLAN_AUTO)
    yield


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("rows,n", [(1, 4096), (300, 4096), (1537, 4096), (4096, 1024), (77, 8192),
                                    (513, 1000)])
@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
def test_host_pipe_matches_oracle(orc, dtype, rows, n, pinned):
    inp = W.generic_rows("add_rms", dtype, rows, n, seed=rows + n)
    x, r = inp["x"], inp["residual"]
    if pinned:
        x, r = x.pin_memory(), r.pin_memory()
    w = inp["w"].cuda()
    rstd = torch.empty(rows, device="cuda")
    ro, y = nrm.add_rms_fwd_host(x, r, w, 1e-6, rstd=rstd)
    gpu = {"residual_out": RN.B.torch_to_np(ro), "y": RN.B.torch_to_np(y),
           "rstd": rstd.cpu().numpy()}
    RN.compare("add_rms", inp, gpu, RN.run_oracle(orc, "add_rms", inp, 1e-6))


def test_host_pipe_in_place_residual_and_repeat(orc):
    inp = W.make_inputs(W.ADD_RMS_BF16_4096x4096, shape=(2500, 4096))
    x = inp["x"].pin_memory()
    ws = nrm.add_rms_fwd_host_workspace(4096, torch.bfloat16)
    w = inp["w"].cuda()
    stream_res = inp["residual"].clone().pin_memory()
    ref = RN.run_oracle(orc, "add_rms", inp, 1e-6)
    ro, y = nrm.add_rms_fwd_host(x, stream_res, w, 1e-6, residual_out=stream_res, workspace=ws)
    assert ro.data_ptr() == stream_res.data_ptr()
    assert np.array_equal(RN.B.torch_to_np(ro), ref["residual_out"])
    RN.T.check_y(2, RN.B.torch_to_np(y), ref["y"], ref["y_wide"], None)
    # a second call on the same workspace, asynchronous, then synchronized
    x2 = torch.zeros_like(x).pin_memory()
    r2 = inp["residual"].clone().pin_memory()
    ro2, y2 = nrm.add_rms_fwd_host(x2, r2, w, 1e-6, workspace=ws, synchronize=False)
    torch.cuda.synchronize()
    inp2 = {"x": x2, "residual": inp["residual"], "w": inp["w"]}
    ref2 = RN.run_oracle(orc, "add_rms", inp2, 1e-6)
    assert np.array_equal(RN.B.torch_to_np(ro2), ref2["residual_out"])
