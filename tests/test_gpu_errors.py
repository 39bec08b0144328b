"""Host-side error handling with a GPU present: invalid calls return a status
and launch nothing.  No test here makes a kernel touch a bad address."""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu

import row_wise_normalization_reduce_gb300 as nrm  # noqa: E402


@pytest.fixture(autouse=True)
def _setup():
    nrm.build()
    nrm.force_plan(nrm.PLAN_AUTO)
    yield
    nrm.set_pointer_checks(False)


def test_inplace_y_rejected():
    x = torch.randn(8, 256, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(nrm.NrmError) as e:
        nrm.ln_fwd(x, out=x)
    assert e.value.status == 4
    with pytest.raises(nrm.NrmError) as e:
        nrm.rms_fwd(x, out=x)
    assert e.value.status == 4


def test_pointer_checks_catch_host_memory():
    lib = nrm.lib()
    dev = torch.empty(8 * 256, device="cuda", dtype=torch.float32)
    host = torch.empty(8 * 256, dtype=torch.float32)
    pinned = torch.empty(8 * 256, dtype=torch.float32).pin_memory()
    nrm.set_pointer_checks(True)
    s = torch.cuda.current_stream().cuda_stream
    for bad in (host.data_ptr(), pinned.data_ptr()):
        st = lib.rms_fwd(bad, None, dev.data_ptr(), None, 8, 256, 1e-6, 0, s)
        assert st == 10, st
        st = lib.rms_fwd(dev.data_ptr(), None, bad, None, 8, 256, 1e-6, 0, s)
        assert st == 10, st
    # device memory passes the check and runs
    out = torch.empty_like(dev)
    assert lib.rms_fwd(dev.data_ptr(), None, out.data_ptr(), None, 8, 256, 1e-6, 0, s) == 0
    torch.cuda.synchronize()


def test_element_misalignment_rejected():
    lib = nrm.lib()
    buf = torch.empty(4096, device="cuda", dtype=torch.uint8)
    p = buf.data_ptr()
    s = torch.cuda.current_stream().cuda_stream
    # bf16 data at an odd byte address
    assert lib.ln_fwd(p + 1, None, None, p + 2048, None, None, 4, 64, 1e-5, 2, s) == 5


def test_bn_workspace_errors():
    x = torch.randn(2, 3, 4, 4, device="cuda")
    small = torch.empty(8, device="cuda", dtype=torch.uint8)
    with pytest.raises(nrm.NrmError) as e:
        nrm.bn_fwd_train(x, workspace=small)
    assert e.value.status == 7
    ws = torch.empty(1024, device="cuda", dtype=torch.uint8)[8:]  # not 16-byte aligned
    with pytest.raises(nrm.NrmError) as e:
        nrm.bn_fwd_train(x, workspace=ws)
    assert e.value.status == 7
    dy = torch.randn_like(x)
    m = torch.zeros(3, device="cuda")
    with pytest.raises(nrm.NrmError) as e:
        nrm.bn_bwd(dy, x, m, m + 1, workspace=small)
    assert e.value.status == 7


def test_status_after_errors_library_still_usable():
    x = torch.randn(4, 512, device="cuda", dtype=torch.float16)
    with pytest.raises(nrm.NrmError):
        nrm.ln_fwd(x, eps=-1.0)
    y, _, _ = nrm.ln_fwd(x)
    torch.cuda.synchronize()
    assert torch.isfinite(y.float()).all()
