"""bn_fwd_train_noalloc, the entry point for callers that cannot allocate device
memory when they call (for instance a runtime that reserves its whole device
memory budget up front, or a component that only receives device pointers).

It keeps the partial statistics in a fixed array inside the library instead of
a caller workspace.  The test calls it through the C ABI with raw device
pointers, twice in a row (the second call finds the array holding the first
call's partials), and compares every output with the workspace entry point
bn_fwd_train on the same inputs, within the tolerances of the other parity
tests (binary32 y: 2e-5 absolute; statistics: 1e-5 relative).

The file name sorts last so that a run stopping at the first failure has run
every other test already; the test also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

OK, TOO_LARGE = 0, 11


def _ptr(t):
    return None if t is None else t.data_ptr()


@pytest.mark.parametrize("shape", [(16, 24, 28, 28), (32, 4, 112, 112)],
                         ids=["cluster_plan", "one_pass_plan"])
def test_noalloc_matches_workspace_entry_point_on_two_calls(shape):
    # (32, 4, 112, 112): planes too large for a cluster's shared memory, so
    # both entry points take the one-pass plan, whose control words live in
    # the library's fixed array for the no-allocation entry point
    import row_wise_normalization_reduce_gb300 as nrm
    from row_wise_normalization_reduce_gb300 import workloads as W

    nrm.build()
    lib = nrm.lib()
    nrm.force_plan(nrm.PLAN_AUTO)
    inp = W.make_inputs(W.BN_F32_32x64x56x56, shape=shape)
    dev = torch.device("cuda", 0)
    x = inp["x"].to(dev)
    g = inp["gamma"].to(dev)
    b = inp["beta"].to(dev)
    batch, c = x.shape[0], x.shape[1]
    hw = x.numel() // (batch * c)
    eps, mom = 1e-5, 0.1
    stream = torch.cuda.current_stream(dev).cuda_stream

    # reference: the workspace entry point, called twice (running stats evolve)
    rm_ref = inp["running_mean"].to(dev)
    rv_ref = inp["running_var"].to(dev)
    refs = []
    for _ in range(2):
        y, sm, sr = nrm.bn_fwd_train(x, g, b, rm_ref, rv_ref, eps, mom)
        torch.cuda.synchronize()
        refs.append((y.clone(), sm.clone(), sr.clone(), rm_ref.clone(), rv_ref.clone()))
    want_plan = nrm.PLAN_TMA if shape[2] * shape[3] < 100 * 100 else nrm.PLAN_PERSIST
    assert nrm.last_plan()[0] == want_plan

    # no-allocation entry point through the C ABI: every buffer passed in
    rm = inp["running_mean"].to(dev)
    rv = inp["running_var"].to(dev)
    y = torch.empty_like(x)
    sm = torch.empty(c, device=dev)
    sr = torch.empty(c, device=dev)
    for call in range(2):
        y.fill_(float("nan"))
        st = lib.bn_fwd_train_noalloc(_ptr(x), _ptr(g), _ptr(b), _ptr(y), _ptr(sm), _ptr(sr),
                                      _ptr(rm), _ptr(rv), batch, c, hw, eps, mom, 0, stream)
        assert st == OK, nrm.status_string(st)
        torch.cuda.synchronize()
        ry, rsm, rsr, rrm, rrv = refs[call]
        assert float((y - ry).abs().max()) <= 2e-5
        for got, want in ((sm, rsm), (sr, rsr), (rm, rrm), (rv, rrv)):
            g64 = got.double().cpu().numpy()
            w64 = want.double().cpu().numpy()
            assert np.all(np.abs(g64 - w64) <= 1e-5 * np.maximum(np.abs(w64), 1e-3))


def test_noalloc_rejects_shapes_beyond_its_capacity():
    import row_wise_normalization_reduce_gb300 as nrm
    nrm.build()
    lib = nrm.lib()
    x = torch.empty(16, device="cuda")
    y = torch.empty(16, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    # batch * C = 65537 planes: refused before anything is launched
    st = lib.bn_fwd_train_noalloc(_ptr(x), None, None, _ptr(y), None, None, None, None,
                                  65537, 1, 2, 1e-5, 0.1, 0, stream)
    assert st == TOO_LARGE
    assert "65536" in nrm.status_string(st)
