"""Chained calls on one stream: each call's input is the previous call's
output, launched back to back (the kernels are programmatic dependent launches
and request their first rows from L2 before waiting for the previous grid),
eagerly and as one CUDA-graph replay.  Every result must equal, bit for bit,
the same chain run with the device synchronized after every call."""
import pytest
import torch

import row_wise_normalization_reduce_gb300 as nrm
from row_wise_normalization_reduce_gb300 import workloads as W

pytestmark = pytest.mark.gpu

STEPS = 6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    nrm.build()
    yield
    nrm.force_plan(nrm.PLAN_AUTO)


def _chain(step, state, sync):
    outs = []
    for _ in range(STEPS):
        state = step(state)
        outs.append(tuple(t.clone() for t in state))
        if sync:
            torch.cuda.synchronize()
    return outs


def _graph_chain(step, state0):
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        step(tuple(t.clone() for t in state0))  # warm-up (plans, caches)
    torch.cuda.synchronize()
    bufs = tuple(t.clone() for t in state0)
    keep = []
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        state = bufs
        for _ in range(STEPS):
            state = step(state)
            keep.append(state)
    g.replay()
    torch.cuda.synchronize()
    return [tuple(t.clone() for t in s) for s in keep]


def _check(step, state0):
    ref = _chain(step, tuple(t.clone() for t in state0), sync=True)
    eager = _chain(step, tuple(t.clone() for t in state0), sync=False)
    torch.cuda.synchronize()
    graph = _graph_chain(step, state0)
    for k in range(STEPS):
        for a, b, c in zip(ref[k], eager[k], graph[k]):
            assert torch.equal(a, b), f"eager step {k}"
            assert torch.equal(a, c), f"graph step {k}"


@pytest.mark.parametrize("shape", [(4096, 4096), (1024, 16384), (300, 1000)])
def test_chained_layernorm(shape):
    inp = W.generic_rows("ln", "bf16", *shape, seed=31)
    g, b = inp["gamma"].cuda(), inp["beta"].cuda()
    _check(lambda s: (nrm.ln_fwd(s[0], g, b, 1e-5)[0],), (inp["x"].cuda(),))


def test_chained_rmsnorm():
    inp = W.generic_rows("rms", "f16", 2048, 4096, seed=32)
    w = inp["w"].cuda()
    _check(lambda s: (nrm.rms_fwd(s[0], w, 1e-6)[0],), (inp["x"].cuda(),))


def test_chained_add_rmsnorm():
    inp = W.generic_rows("add_rms", "bf16", 4096, 4096, seed=33)
    w = inp["w"].cuda()

    def step(s):
        ro, y, _ = nrm.add_rms_fwd(s[0], s[1], w, 1e-6)
        return (y, ro)
    _check(step, (inp["x"].cuda(), inp["residual"].cuda()))


def test_chained_softmax():
    x = (4 * torch.randn(4096, 4096, generator=torch.Generator().manual_seed(34))).to(torch.bfloat16)
    _check(lambda s: (nrm.softmax_fwd(s[0])[0],), (x.cuda(),))


@pytest.mark.parametrize("plan", [nrm.PLAN_AUTO, nrm.PLAN_PERSIST], ids=["auto", "flow"])
@pytest.mark.parametrize("shape", [(32, 64, 56, 56), (4, 16, 112, 112)])
def test_chained_batchnorm_forward(shape, plan):
    inp = W.make_inputs(W.BN_F32_32x64x56x56, shape=shape)
    g, b = inp["gamma"].cuda(), inp["beta"].cuda()
    nrm.force_plan(plan)
    try:
        _check(lambda s: (nrm.bn_fwd_train(s[0], g, b, None, None, 1e-5, 0.1)[0],), (inp["x"].cuda(),))
    finally:
        nrm.force_plan(nrm.PLAN_AUTO)


def test_chained_batchnorm_backward():
    inp = W.make_inputs(W.BN_BWD_F32_32x64x56x56, shape=(4, 16, 112, 112))
    x, sm, sr, g = (inp[k].cuda() for k in ("x", "save_mean", "save_rstd", "gamma"))
    _check(lambda s: (nrm.bn_bwd(s[0], x, sm, sr, g)[0],), (inp["dy"].cuda(),))
