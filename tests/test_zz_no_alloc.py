"""bn_fwd_train_noalloc, the entry point for callers that cannot allocate device
memory when they call (for instance a runtime that reserves its whole device
memory budget up front, or a component that only receives device pointers).

It keeps the partial statistics in a fixed array inside the library instead of
a caller workspace.  The tests call it through the C ABI with raw device
pointers, twice in a row on different inputs (the second call finds the array
holding the first call's partials), on every BatchNorm plan that can use the
array, and check every output against the CPU oracle with the tolerances of
the other parity tests (binary32 y: 2e-5 absolute; 16-bit y: 1 ulp;
statistics: 1e-5 relative) and against the workspace entry point bn_fwd_train
on the same inputs.  They also check that it honours the wait limit (its
bounded waits give up and raise the fault bit) and the pointer checks.

The file name sorts last so that a run stopping at the first failure has run
every other test already; the tests also pass alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import runners as RN

pytestmark = pytest.mark.gpu

OK, POINTER, TOO_LARGE = 0, 10, 11
EPS, MOM = 1e-5, 0.1


def _ptr(t):
    return None if t is None else t.data_ptr()


@pytest.fixture(autouse=True)
def _restore():
    import row_wise_normalization_reduce_gb300 as nrm
    nrm.build()
    nrm.force_plan(nrm.PLAN_AUTO)
    yield
    nrm.force_plan(nrm.PLAN_AUTO)
    nrm.set_pointer_checks(False)


def _second_input(inp):
    """A second input set of the same shape with other values (derived on the
    CPU), so that stale partials of the first call would show."""
    out = dict(inp)
    x = inp["x"].double()
    out["x"] = (x * 0.5 - 1.25).to(inp["x"].dtype)
    return out


def _noalloc(lib, d, dtype_code):
    """One call through the C ABI with every buffer passed in; returns the
    outputs (running statistics start from the inputs' values)."""
    x = d["x"]
    batch, c = x.shape[0], x.shape[1]
    hw = x.numel() // (batch * c)
    y = torch.full_like(x, float("nan"))
    sm = torch.full((c,), float("nan"), device=x.device)
    sr = torch.full((c,), float("nan"), device=x.device)
    rm = d["running_mean"].clone()
    rv = d["running_var"].clone()
    st = lib.bn_fwd_train_noalloc(_ptr(x), _ptr(d.get("gamma")), _ptr(d.get("beta")), _ptr(y),
                                  _ptr(sm), _ptr(sr), _ptr(rm), _ptr(rv), batch, c, hw, EPS, MOM,
                                  dtype_code, torch.cuda.current_stream().cuda_stream)
    return st, {"y": y, "save_mean": sm, "save_rstd": sr, "running_mean": rm, "running_var": rv}


def _np(out):
    import bits as B
    return {k: B.torch_to_np(v.cpu()) for k, v in out.items()}


# (shape, dtype, forced row plan naming the BatchNorm plan, plan that must run)
CASES = [
    ((16, 24, 28, 28), "f32", "auto", "tma"),         # cluster per channel
    ((32, 4, 112, 112), "f32", "auto", "persist"),    # one-pass (control words in the array)
    ((16, 24, 28, 28), "f32", "cta", "cta"),          # streaming: per-chunk partials
    ((16, 24, 28, 28), "bf16", "generic", "generic"),  # scalar: per-plane partials
    ((8, 6, 40, 56), "f16", "persist", "persist"),    # one-pass, 16-bit, several chunks
    # batch * C * chunks of 1024 packs per plane > 65536: the streaming plan
    # is left out; the cluster plan cannot hold 64 planes of 4100 values, so
    # the one-pass plan (one 2048-pack item per plane) runs on the array
    ((64, 520, 41, 100), "f32", "auto", "persist"),
    # the same shape forced onto the streaming plan: it falls back as well
    ((64, 520, 41, 100), "f32", "cta", "persist"),
]


@pytest.mark.parametrize("shape,dtype,force,want", CASES,
                         ids=[f"{c[2]}-{c[1]}-{'x'.join(map(str, c[0]))}" for c in CASES])
def test_noalloc_two_calls_against_oracle_and_workspace_entry_point(orc, shape, dtype, force,
                                                                     want):
    import row_wise_normalization_reduce_gb300 as nrm
    from row_wise_normalization_reduce_gb300 import workloads as W

    lib = nrm.lib()
    codes = {v: k for k, v in nrm.PLAN_NAMES.items()}
    nrm.force_plan(codes[force])
    dev = torch.device("cuda", 0)
    inp_a = W.make_inputs(W.BN_F32_32x64x56x56, shape=shape, dtype=dtype)
    big = shape[0] * shape[1] > 20000
    chans = [0, shape[1] // 2, shape[1] - 1]
    for call, inp in enumerate((inp_a, _second_input(inp_a))):
        d = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
        st, got = _noalloc(lib, d, {"f32": 0, "f16": 1, "bf16": 2}[dtype])
        assert st == OK, nrm.status_string(st)
        torch.cuda.synchronize()
        assert nrm.PLAN_NAMES[nrm.last_plan()[0]] == want, (call, nrm.last_plan())
        # the workspace entry point on the same inputs, forced onto the same plan
        nrm.force_plan(codes[want])
        rm, rv = d["running_mean"].clone(), d["running_var"].clone()
        y, sm, sr = nrm.bn_fwd_train(d["x"], d.get("gamma"), d.get("beta"), rm, rv, EPS, MOM)
        torch.cuda.synchronize()
        assert nrm.PLAN_NAMES[nrm.last_plan()[0]] == want
        nrm.force_plan(codes[force])
        ref_ws = {"y": y, "save_mean": sm, "save_rstd": sr, "running_mean": rm, "running_var": rv}
        for k, v in got.items():
            w_ = ref_ws[k]
            assert not torch.isnan(v).any(), k
            if dtype == "f32" or k != "y":
                err = (v.double() - w_.double()).abs()
                lim = 2e-5 if k == "y" else 1e-5 * w_.double().abs().clamp_min(1e-3)
                assert bool((err <= lim).all()), (call, k)
        # the oracle on the same inputs (sampled channels for the large case;
        # channels are independent)
        g_np = _np(got)
        if big:
            sub = RN.select_channels("bn", inp, chans)
            ref = RN.run_oracle(orc, "bn", sub, EPS, MOM)
            RN.compare("bn", sub, RN.slice_gpu_channels(g_np, chans), ref)
        else:
            RN.compare("bn", inp, g_np, RN.run_oracle(orc, "bn", inp, EPS, MOM))


@pytest.mark.parametrize("force,want", [("auto", "tma"), ("persist", "persist")])
def test_noalloc_bounded_waits_give_up_and_report(orc, force, want):
    # wait limit 0: every bounded wait of the cluster plan (its bulk copies)
    # and of the one-pass plan (its statistics polls) gives up at once; the
    # kernel raises the fault bit and ends, and the next call is correct
    import row_wise_normalization_reduce_gb300 as nrm
    from row_wise_normalization_reduce_gb300 import workloads as W

    lib = nrm.lib()
    codes = {v: k for k, v in nrm.PLAN_NAMES.items()}
    nrm.force_plan(codes[force])
    inp = W.make_inputs(W.BN_F32_32x64x56x56, shape=(8, 16, 28, 28))
    d = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    assert nrm.device_fault(clear=True) == 0
    old = nrm.set_wait_limit(0)
    try:
        st, _ = _noalloc(lib, d, 0)
        torch.cuda.synchronize()
        bits = nrm.device_fault(clear=True)
    finally:
        nrm.set_wait_limit(old)
    assert st == OK
    assert nrm.PLAN_NAMES[nrm.last_plan()[0]] == want
    assert bits & 1, bits
    st, got = _noalloc(lib, d, 0)
    assert st == OK
    torch.cuda.synchronize()
    assert nrm.device_fault(clear=True) == 0
    RN.compare("bn", inp, _np(got), RN.run_oracle(orc, "bn", inp, EPS, MOM))


def test_noalloc_rejects_host_memory_and_bad_tensors():
    import row_wise_normalization_reduce_gb300 as nrm
    lib = nrm.lib()
    x = torch.randn(4, 3, 8, 8, device="cuda")
    y = torch.empty_like(x)
    sm = torch.empty(3, device="cuda")
    sr = torch.empty(3, device="cuda")
    host = torch.empty(3)
    s = torch.cuda.current_stream().cuda_stream
    nrm.set_pointer_checks(True)
    for pos in range(4):  # a host pointer as gamma, save_mean, save_rstd or running_mean
        ptrs = [None, _ptr(sm), _ptr(sr), None]
        ptrs[pos] = host.data_ptr()
        st = lib.bn_fwd_train_noalloc(_ptr(x), ptrs[0], None, _ptr(y), ptrs[1], ptrs[2], ptrs[3],
                                      None, 4, 3, 64, EPS, MOM, 0, s)
        assert st == POINTER, (pos, st)
    nrm.set_pointer_checks(False)
    # the Python wrapper checks tensors before the call
    with pytest.raises(ValueError):
        nrm.bn_fwd_train_noalloc(x, out=y, save_mean=host, save_rstd=sr)
    with pytest.raises(ValueError):
        nrm.bn_fwd_train_noalloc(x, torch.ones(3), out=y, save_mean=sm, save_rstd=sr)
    with pytest.raises(ValueError):
        nrm.bn_fwd_train_noalloc(x, out=torch.empty(4, 3, 8, 7, device="cuda"), save_mean=sm,
                                 save_rstd=sr)
    with pytest.raises(ValueError):
        nrm.bn_fwd_train_noalloc(x, out=y, save_mean=sm, save_rstd=None)


def test_noalloc_rejects_shapes_beyond_its_capacity():
    import row_wise_normalization_reduce_gb300 as nrm
    lib = nrm.lib()
    x = torch.empty(16, device="cuda")
    y = torch.empty(16, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    # batch * C = 65537 planes: refused before anything is launched
    st = lib.bn_fwd_train_noalloc(_ptr(x), None, None, _ptr(y), None, None, None, None,
                                  65537, 1, 2, 1e-5, 0.1, 0, stream)
    assert st == TOO_LARGE
    assert "65536" in nrm.status_string(st)
