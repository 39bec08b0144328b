"""BatchNorm beyond the binary32 training forward: 16-bit training forward,
inference forward (running statistics) and training backward, on every plan,
over shapes that cover one plane, planes narrower than a 16-byte pack, odd
H*W, many small planes and multi-plane channels; against the CPU oracle."""
import dataclasses

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
    yield
    nrm.force_plan(nrm.PLAN_AUTO)


TRAIN_PLANS = [nrm.PLAN_AUTO, nrm.PLAN_CTA, nrm.PLAN_TMA, nrm.PLAN_GENERIC, nrm.PLAN_PERSIST]
TRAIN_IDS = ["auto", "stream", "cluster", "scalar", "flow"]
TWO_PLANS = [nrm.PLAN_AUTO, nrm.PLAN_GENERIC]
TWO_IDS = ["auto", "scalar"]
SHAPES = [(1, 3, 5, 5), (2, 4, 3, 3), (4, 8, 1, 1), (2, 3, 4, 8), (3, 5, 13, 11), (8, 16, 28, 28),
          (5, 7, 20, 20), (2, 64, 4, 4), (32, 4, 56, 56)]


@pytest.mark.parametrize("plan", TRAIN_PLANS, ids=TRAIN_IDS)
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("shape", SHAPES)
def test_bn_train_half_types(orc, shape, dtype, plan):
    inp = W.make_inputs(W.BN_F32_32x64x56x56, shape=shape, dtype=dtype)
    nrm.force_plan(plan)
    gpu = RN.run_gpu("bn", inp, 1e-5, 0.1)
    RN.compare("bn", inp, gpu, RN.run_oracle(orc, "bn", inp, 1e-5, 0.1))


@pytest.mark.parametrize("plan", TWO_PLANS, ids=TWO_IDS)
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("shape", SHAPES + [(1, 1, 1, 1), (4, 8, 7, 7), (3, 2, 1, 33)])
def test_bn_infer_shapes(orc, shape, dtype, plan):
    inp = W.make_inputs(W.BN_INFER_F32_32x64x56x56, shape=shape, dtype=dtype)
    nrm.force_plan(plan)
    gpu = RN.run_gpu("bn_infer", inp, 1e-5)
    RN.compare("bn_infer", inp, gpu, RN.run_oracle(orc, "bn_infer", inp, 1e-5))


@pytest.mark.parametrize("plan", TWO_PLANS, ids=TWO_IDS)
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("shape", SHAPES + [(1, 1, 1, 1), (1, 2, 1, 5), (4, 8, 7, 7)])
def test_bn_bwd_shapes(orc, shape, dtype, plan):
    inp = W.make_inputs(W.BN_BWD_F32_32x64x56x56, shape=shape, dtype=dtype)
    nrm.force_plan(plan)
    gpu = RN.run_gpu("bn_bwd", inp, 1e-5)
    RN.compare("bn_bwd", inp, gpu, RN.run_oracle(orc, "bn_bwd", inp, 1e-5))


def test_bn_infer_empty_batch_and_no_affine(orc):
    nrm.force_plan(nrm.PLAN_AUTO)
    inp = W.make_inputs(W.BN_INFER_F32_32x64x56x56, shape=(3, 6, 10, 10))
    d = {k: v.cuda() for k, v in inp.items()}
    y = nrm.bn_fwd_infer(d["x"], d["running_mean"], d["running_var"])
    torch.cuda.synchronize()
    n = RN.to_np(inp)
    ref = orc.batchnorm_infer(0, n["x"], n["running_mean"], n["running_var"], wide=True)
    assert np.max(np.abs(y.cpu().numpy().reshape(ref["y_wide"].shape) - ref["y_wide"])) <= 2e-5
    empty = torch.empty(0, 6, 10, 10, device="cuda")
    assert nrm.bn_fwd_infer(empty, d["running_mean"], d["running_var"]).numel() == 0


def test_bn_bwd_without_gamma_and_sums(orc):
    nrm.force_plan(nrm.PLAN_AUTO)
    inp = W.make_inputs(W.BN_BWD_F32_32x64x56x56, shape=(4, 5, 12, 12))
    inp["gamma"] = None
    gpu = RN.run_gpu("bn_bwd", inp, 1e-5)
    RN.compare("bn_bwd", inp, gpu, RN.run_oracle(orc, "bn_bwd", inp, 1e-5))
    # dgamma / dbeta not written when absent: call the C ABI with NULLs
    d = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    dx = torch.full_like(d["x"], float("nan"))
    ws = torch.empty(nrm.bn_bwd_workspace_size(4, 5, 144), dtype=torch.uint8, device="cuda")
    st = nrm.lib().bn_bwd(d["dy"].data_ptr(), d["x"].data_ptr(), None, d["save_mean"].data_ptr(),
                          d["save_rstd"].data_ptr(), dx.data_ptr(), None, None, 4, 5, 144, 0,
                          ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert np.array_equal(dx.cpu().numpy(), gpu["dx"])


@pytest.mark.parametrize("w", [W.BN_BWD_F32_32x64x56x56, W.BN_INFER_F32_32x64x56x56],
                         ids=lambda w: w.name)
def test_bn_plans_agree_and_repeat(w):
    inp = W.make_inputs(w, shape=(16, 8, 28, 28))
    outs = []
    for plan in (nrm.PLAN_AUTO, nrm.PLAN_AUTO, nrm.PLAN_GENERIC):
        nrm.force_plan(plan)
        outs.append(RN.run_gpu(w.op, inp, 1e-5))
    for k in outs[0]:
        assert (outs[0][k] == outs[1][k]).all(), k
        a, b = outs[0][k].astype(np.float64), outs[2][k].astype(np.float64)
        assert np.max(np.abs(a - b)) <= 1e-4 * max(1.0, float(np.max(np.abs(a)))), k


def test_bn_forward_then_backward_on_gpu():
    # a property that holds for any data: with the batch's own statistics the
    # gradient dx sums to zero over each channel (sum of xhat is zero)
    nrm.force_plan(nrm.PLAN_AUTO)
    inp = W.make_inputs(W.BN_F32_32x64x56x56, shape=(8, 16, 28, 28))
    x = inp["x"].cuda()
    g = inp["gamma"].cuda()
    y, sm, sr = nrm.bn_fwd_train(x, g, inp["beta"].cuda(), None, None, 1e-5, 0.1)
    dy = torch.randn(x.shape, generator=torch.Generator().manual_seed(5)).cuda()
    dx, dg, db = nrm.bn_bwd(dy, x, sm, sr, g)
    torch.cuda.synchronize()
    s = dx.double().sum(dim=(0, 2, 3)).abs()
    assert torch.all(s <= 1e-4 * dx.double().abs().sum(dim=(0, 2, 3)))
    assert torch.allclose(db.double(), dy.double().sum(dim=(0, 2, 3)), rtol=1e-5, atol=1e-3)


@pytest.mark.parametrize("op", ["bn", "bn_bwd"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("group_bytes", [0, 1], ids=["default_groups", "one_channel_groups"])
@pytest.mark.parametrize("shape", [(2, 5, 64, 80), (1, 2, 96, 96), (2, 3, 70, 70), (3, 4, 40, 200)])
def test_bn_stream_chunks_and_groups(orc, shape, group_bytes, dtype, op):
    # planes longer than one 1024-pack unit (several chunks per plane, the
    # last one shorter where the plane does not divide evenly), and channel
    # groups down to one channel per group (two launches per channel)
    w = W.BN_F32_32x64x56x56 if op == "bn" else W.BN_BWD_F32_32x64x56x56
    inp = W.make_inputs(w, shape=shape, dtype=dtype)
    nrm.force_plan(nrm.PLAN_CTA)
    old = nrm.set_bn_group_bytes(group_bytes)
    try:
        gpu = RN.run_gpu(op, inp, 1e-5, 0.1)
        again = RN.run_gpu(op, inp, 1e-5, 0.1)
    finally:
        nrm.set_bn_group_bytes(old)
    for k in gpu:
        assert (gpu[k] == again[k]).all(), k
    RN.compare(op, inp, gpu, RN.run_oracle(orc, op, inp, 1e-5, 0.1))


@pytest.mark.parametrize("packs", [0, 4, 8], ids=["auto_packs", "packs4", "packs8"])
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("shape", [(2, 5, 64, 80), (1, 2, 96, 96), (2, 3, 70, 70), (3, 4, 40, 200),
                                   (1, 1, 64, 64), (2, 1, 200, 200), (4, 40, 32, 32),
                                   (64, 64, 16, 16), (32, 64, 56, 56)])
def test_bn_flow_chunks_and_lag(orc, shape, dtype, packs):
    # the one-pass plan at four and eight packs per thread: several chunks per
    # plane (the last one shorter where the plane does not divide evenly), a
    # single channel (every statistics item before any normalize item), more
    # items than resident CTAs (normalize items interleaved with later
    # channels' statistics); bitwise repeatable; layouts it cannot take fall
    # back to another plan
    inp = W.make_inputs(W.BN_F32_32x64x56x56, shape=shape, dtype=dtype)
    nrm.force_plan(nrm.PLAN_PERSIST, 0, packs)
    gpu = RN.run_gpu("bn", inp, 1e-5, 0.1)
    hw = shape[2] * shape[3]
    packed = hw % (4 if dtype == "f32" else 8) == 0
    assert (nrm.last_plan()[0] == nrm.PLAN_PERSIST) == packed
    again = RN.run_gpu("bn", inp, 1e-5, 0.1)
    for k in gpu:
        assert (gpu[k] == again[k]).all(), k
    RN.compare("bn", inp, gpu, RN.run_oracle(orc, "bn", inp, 1e-5, 0.1))


def test_bn_flow_ignores_workspace_contents(orc):
    # the control words live in the caller's workspace and are reset by the
    # call itself: a workspace full of 0xFF bytes gives the same result
    inp = W.make_inputs(W.BN_F32_32x64x56x56, shape=(6, 10, 40, 40))
    nrm.force_plan(nrm.PLAN_PERSIST)
    ref = RN.run_gpu("bn", inp, 1e-5, 0.1)
    x, g, b = inp["x"].cuda(), inp["gamma"].cuda(), inp["beta"].cuda()
    need = nrm.bn_fwd_train_workspace_size(6, 10, 1600)
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")
    for _ in range(2):
        y, sm, sr = nrm.bn_fwd_train(x, g, b, None, None, 1e-5, 0.1, workspace=ws)
        torch.cuda.synchronize()
        assert nrm.last_plan()[0] == nrm.PLAN_PERSIST
        assert np.array_equal(y.cpu().numpy(), ref["y"])
        assert np.array_equal(sm.cpu().numpy(), ref["save_mean"])
        assert np.array_equal(sr.cpu().numpy(), ref["save_rstd"])


def test_bn_flow_wait_give_up_path(orc):
    # wait limit 0: every normalize item gives up its wait for the channel's
    # statistics at once; the kernel must raise the fault bit and still end,
    # and the next call must be correct
    inp = W.make_inputs(W.BN_F32_32x64x56x56, shape=(8, 16, 28, 28))
    nrm.force_plan(nrm.PLAN_PERSIST)
    x = inp["x"].cuda()
    assert nrm.device_fault(clear=True) == 0
    old = nrm.set_wait_limit(0)
    try:
        nrm.bn_fwd_train(x, None, None, None, None, 1e-5, 0.1)
        bits = nrm.device_fault(clear=True)
    finally:
        nrm.set_wait_limit(old)
    assert nrm.last_plan()[0] == nrm.PLAN_PERSIST
    assert bits == 1, bits
    gpu = RN.run_gpu("bn", inp, 1e-5, 0.1)
    RN.compare("bn", inp, gpu, RN.run_oracle(orc, "bn", inp, 1e-5, 0.1))
    assert nrm.device_fault(clear=True) == 0


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("shape", [(2, 5, 64, 80), (1, 2, 96, 96), (2, 3, 70, 70), (3, 4, 40, 200),
                                   (1, 1, 64, 64), (2, 1, 200, 200), (4, 40, 32, 32),
                                   (64, 64, 16, 16), (16, 8, 56, 56)])
def test_bn_bwd_flow_chunks_and_lag(orc, shape, dtype):
    # the one-pass backward: several chunks per plane, a single channel, more
    # items than resident CTAs; bitwise repeatable; layouts it cannot take
    # fall back to another plan
    inp = W.make_inputs(W.BN_BWD_F32_32x64x56x56, shape=shape, dtype=dtype)
    nrm.force_plan(nrm.PLAN_PERSIST)
    gpu = RN.run_gpu("bn_bwd", inp, 1e-5)
    hw = shape[2] * shape[3]
    packed = hw % (4 if dtype == "f32" else 8) == 0
    assert (nrm.last_plan()[0] == nrm.PLAN_PERSIST) == packed
    again = RN.run_gpu("bn_bwd", inp, 1e-5)
    for k in gpu:
        assert (gpu[k] == again[k]).all(), k
    RN.compare("bn_bwd", inp, gpu, RN.run_oracle(orc, "bn_bwd", inp, 1e-5))


def test_bn_bwd_flow_wait_give_up_path(orc):
    # wait limit 0: every wait of the one-pass backward gives up at once; the
    # kernel raises the fault bit and ends, and the next call is correct
    inp = W.make_inputs(W.BN_BWD_F32_32x64x56x56, shape=(8, 16, 40, 40))
    nrm.force_plan(nrm.PLAN_PERSIST)
    d = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    assert nrm.device_fault(clear=True) == 0
    old = nrm.set_wait_limit(0)
    try:
        nrm.bn_bwd(d["dy"], d["x"], d["save_mean"], d["save_rstd"], d["gamma"])
        bits = nrm.device_fault(clear=True)
    finally:
        nrm.set_wait_limit(old)
    assert nrm.last_plan()[0] == nrm.PLAN_PERSIST
    assert bits == 1, bits
    gpu = RN.run_gpu("bn_bwd", inp, 1e-5)
    RN.compare("bn_bwd", inp, gpu, RN.run_oracle(orc, "bn_bwd", inp, 1e-5))
    assert nrm.device_fault(clear=True) == 0
