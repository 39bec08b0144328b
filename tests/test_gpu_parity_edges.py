"""GPU parity on edge cases: row lengths around every pack and plan boundary,
empty and single rows, misaligned pointers (scalar path), absent parameters,
constant rows, every plan forced on the same inputs, 3-D inputs, guard bands
around outputs, BatchNorm corner shapes.  All compared element by element with
the CPU oracle."""
import numpy as np
import pytest
import torch

import bits as B
import runners as RN
from row_wise_normalization_reduce_gb300 import workloads as W

pytestmark = pytest.mark.gpu

import row_wise_normalization_reduce_gb300 as nrm  # noqa: E402

DTYPES = ["f32", "f16", "bf16"]


@pytest.fixture(autouse=True)
def _auto_plan():
    nrm.build()
    nrm.force_plan(nrm.PLAN_AUTO)
    yield
    nrm.force_plan(nrm.PLAN_AUTO)


def _check(orc, op, inp, eps=1e-5):
    gpu = RN.run_gpu(op, inp, eps)
    ref = RN.run_oracle(orc, op, inp, eps)
    return RN.compare(op, inp, gpu, ref)


@pytest.mark.parametrize("op", ["ln", "rms", "add_rms"])
@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("n", [1, 2, 3, 7, 8, 255, 256, 1000, 1024, 4096, 8192, 16384, 32768,
                               65536])
def test_row_lengths(orc, op, dt, n):
    rows = 3 if n >= 16384 else 37
    inp = W.generic_rows(op, dt, rows, n, seed=n + 17, scale=2.0, shift=1.0)
    _check(orc, op, inp)


@pytest.mark.parametrize("op", ["ln", "rms", "add_rms"])
@pytest.mark.parametrize("rows", [0, 1, 3, 64, 4097])
def test_row_counts(orc, op, rows):
    inp = W.generic_rows(op, "bf16", rows, 512, seed=rows + 5)
    if rows == 0:
        d = {k: v.cuda() for k, v in inp.items()}
        if op == "ln":
            y, m, r = nrm.ln_fwd(d["x"], d["gamma"], d["beta"])
            assert y.numel() == 0
        elif op == "rms":
            y, _ = nrm.rms_fwd(d["x"], d["w"])
        else:
            nrm.add_rms_fwd(d["x"], d["residual"], d["w"])
        return
    _check(orc, op, inp)


PLANS = [(nrm.PLAN_GENERIC, 128, 0), (nrm.PLAN_GENERIC, 256, 0), (nrm.PLAN_GENERIC, 512, 0),
         (nrm.PLAN_WARP, 128, 8), (nrm.PLAN_CTA, 128, 2), (nrm.PLAN_CTA, 256, 1),
         (nrm.PLAN_CTA, 256, 2), (nrm.PLAN_CTA, 512, 1), (nrm.PLAN_CTA, 1024, 1),
         (nrm.PLAN_CTA, 256, 4), (nrm.PLAN_CTA, 512, 4), (nrm.PLAN_CTA, 1024, 4),
         (nrm.PLAN_CTA, 1024, 2), (nrm.PLAN_CTA, 512, 2),
         (nrm.PLAN_TMA, 128, 4, 2, 1), (nrm.PLAN_TMA, 128, 4, 3, 8), (nrm.PLAN_TMA, 256, 2, 0, 0),
         (nrm.PLAN_TMA, 256, 4, 5, 2), (nrm.PLAN_TMA, 512, 4, 2, 2), (nrm.PLAN_TMA, 128, 8, 16, 1),
         (nrm.PLAN_PERSIST, 256, 1), (nrm.PLAN_PERSIST, 128, 4), (nrm.PLAN_PERSIST, 1024, 2),
         (nrm.PLAN_WRAW, 256, 8), (nrm.PLAN_WRAW, 512, 16), (nrm.PLAN_WRAW, 256, 32)]


@pytest.mark.parametrize("op", ["ln", "rms", "add_rms"])
@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("plan", PLANS,
                         ids=lambda p: f"{nrm.PLAN_NAMES[p[0]]}{p[1]}x{p[2]}" + (
                             f"s{p[3]}g{p[4]}" if len(p) > 3 else ""))
def test_forced_plans(orc, op, dt, plan):
    # N = 1000 elements: a ragged number of packs for every dtype that fits
    # every plan above (fp32: 250 packs, 16-bit: 125 packs)
    n = 1000 if dt == "f32" else 2000
    if plan[0] == nrm.PLAN_WARP:
        n = 1000 if dt == "f32" else 1000
    inp = W.generic_rows(op, dt, 67, n, seed=3, scale=1.5, shift=0.5)
    nrm.force_plan(*plan)
    _check(orc, op, inp)
    got = nrm.last_plan()
    assert got[0] == plan[0]


@pytest.mark.parametrize("op", ["ln", "rms", "add_rms"])
@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("shape", [(512, 4), (1024, 2)], ids=lambda c: f"{c[0]}x{c[1]}")
def test_persist_exact_rows(orc, op, dt, shape):
    # rows of exactly THREADS x PACKS packs (every thread's packs in range);
    # 400 rows give every persistent CTA two or three rows
    th, pk = shape
    n = th * pk * (4 if dt == "f32" else 8)
    inp = W.generic_rows(op, dt, 400, n, seed=th + pk, scale=1.5, shift=0.5)
    nrm.force_plan(nrm.PLAN_PERSIST, th, pk)
    _check(orc, op, inp)
    assert nrm.last_plan()[0] == nrm.PLAN_PERSIST


# cluster split (threads, packs per thread, CTAs per cluster): every compiled
# instance
CLUSTER_SHAPES = [(128, 1, 2), (128, 1, 4), (128, 2, 2), (128, 2, 4), (128, 4, 2), (128, 4, 4),
                  (128, 4, 8), (256, 4, 2)]


@pytest.mark.parametrize("op", ["ln", "rms", "add_rms"])
@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("shape", CLUSTER_SHAPES, ids=lambda c: f"{c[0]}x{c[1]}c{c[2]}")
@pytest.mark.parametrize("fill", ["full", "ragged"])
def test_cluster_split_plans(orc, op, dt, shape, fill):
    # one row over a cluster of CTAs: every slice exactly THREADS x PACKS packs
    # (no bounds tests) or 37 packs short of it (bounds tests in every CTA)
    threads, packs, cs = shape
    v = 4 if dt == "f32" else 8
    s = threads * packs - (0 if fill == "full" else min(37, threads * packs - 1))
    inp = W.generic_rows(op, dt, 45, s * cs * v, seed=cs * 100 + s, scale=1.7, shift=-0.6)
    nrm.force_plan(nrm.PLAN_CLUSTER, threads, packs, 0, cs)
    _check(orc, op, inp)
    assert nrm.last_plan() == (nrm.PLAN_CLUSTER, threads, packs, 0, cs)


def test_cluster_split_refuses_rows_it_cannot_split():
    # 1000 binary32 values are 250 packs: not a multiple of 4 or 8 CTAs
    x = torch.randn(4, 1000, device="cuda")
    for cs in (4, 8):
        nrm.force_plan(nrm.PLAN_CLUSTER, 128, 2, 0, cs)
        with pytest.raises(nrm.NrmError) as e:
            nrm.ln_fwd(x)
        assert e.value.status == 6


@pytest.mark.parametrize("op", ["ln", "rms", "add_rms"])
@pytest.mark.parametrize("dt,threads,packs,groups", [("bf16", 128, 4, 4), ("f32", 256, 4, 2),
                                                     ("f16", 256, 2, 1), ("bf16", 128, 4, 8)])
@pytest.mark.parametrize("stages", [2, 3, 5])
def test_tma_pipeline_many_rows_per_cta(orc, op, dt, threads, packs, groups, stages):
    # 3001 rows over at most a few hundred row groups: every group streams many
    # rows through its ring, so stages are refilled, barrier phases alternate
    # and groups claim rows from their CTA's range until it runs out.
    inp = W.generic_rows(op, dt, 3001, 4096, seed=stages, scale=1.3, shift=-0.4)
    try:
        nrm.force_plan(nrm.PLAN_TMA, threads, packs, stages, groups)
        _check(orc, op, inp)
    except nrm.NrmError as e:
        # only a shared-memory budget overflow may refuse this combination
        assert e.status == 6
        pytest.skip("stages x groups exceed the shared memory of one CTA")
    assert nrm.last_plan() == (nrm.PLAN_TMA, threads, packs, stages, groups)


@pytest.mark.parametrize("op", ["ln", "rms", "add_rms"])
@pytest.mark.parametrize("dt,threads,packs", [("bf16", 256, 2), ("f32", 512, 2), ("f16", 128, 4)])
def test_persist_many_rows_per_cta(orc, op, dt, threads, packs):
    # 3001 rows over the resident CTAs: each CTA prefetches row r + G while it
    # reduces row r, several times over, and ends on a ragged last round.
    inp = W.generic_rows(op, dt, 3001, 4096, seed=31, scale=0.7, shift=2.0)
    nrm.force_plan(nrm.PLAN_PERSIST, threads, packs)
    _check(orc, op, inp)
    assert nrm.last_plan()[:3] == (nrm.PLAN_PERSIST, threads, packs)


@pytest.mark.parametrize("op", ["ln", "rms", "add_rms"])
@pytest.mark.parametrize("dt,n", [("bf16", 4096), ("f32", 2048), ("f16", 4096), ("bf16", 3000)])
def test_wraw_many_rows(orc, op, dt, n):
    inp = W.generic_rows(op, dt, 1501, n, seed=41, scale=1.1, shift=-0.3)
    nrm.force_plan(nrm.PLAN_WRAW, 256, 16)
    _check(orc, op, inp)
    assert nrm.last_plan()[:3] == (nrm.PLAN_WRAW, 256, 16)


def test_tma_wait_give_up_path(orc):
    # With a wait limit of 0 every bulk-copy wait gives up at once: the kernel
    # must flag the fault, drain its copies and return (outputs undefined), and
    # the next call with the normal limit must be correct again.
    inp = W.generic_rows("add_rms", "bf16", 900, 4096, seed=77)
    d = {k: v.cuda() for k, v in inp.items()}
    nrm.force_plan(nrm.PLAN_TMA, 128, 4, 3, 4)
    assert nrm.device_fault(clear=True) == 0
    old = nrm.set_wait_limit(0)
    try:
        nrm.add_rms_fwd(d["x"], d["residual"], d["w"], 1e-6)
        bits = nrm.device_fault(clear=True)
    finally:
        nrm.set_wait_limit(old)
    assert bits == 1, bits            # gave up waiting, drained cleanly
    _check(orc, "add_rms", inp, eps=1e-6)
    assert nrm.device_fault(clear=True) == 0


def test_forced_plan_that_cannot_run():
    nrm.force_plan(nrm.PLAN_WARP, 128, 1)
    x = torch.randn(4, 4096, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(nrm.NrmError) as e:
        nrm.rms_fwd(x)
    assert e.value.status == 6


@pytest.mark.parametrize("op", ["ln", "rms", "add_rms"])
@pytest.mark.parametrize("dt", DTYPES)
def test_misaligned_pointers_use_scalar_path(orc, op, dt):
    rows, n = 9, 512
    inp = W.generic_rows(op, dt, rows, n, seed=11)
    d = {}
    for k, v in inp.items():
        buf = torch.empty(v.numel() + 1, dtype=v.dtype, device="cuda")
        view = buf[1:].view(v.shape)
        view.copy_(v.cuda())
        d[k] = view
    if op == "ln":
        y, mean, rstd = nrm.ln_fwd(d["x"], d["gamma"], d["beta"], 1e-5)
        gpu = {"y": y, "mean": mean, "rstd": rstd}
    elif op == "rms":
        y, rstd = nrm.rms_fwd(d["x"], d["w"], 1e-5, want_stats=True)
        gpu = {"y": y, "rstd": rstd}
    else:
        ro, y, rstd = nrm.add_rms_fwd(d["x"], d["residual"], d["w"], 1e-5, want_stats=True)
        gpu = {"residual_out": ro, "y": y, "rstd": rstd}
    assert nrm.last_plan()[0] == nrm.PLAN_GENERIC
    torch.cuda.synchronize()
    gpu = {k: B.torch_to_np(v.cpu()) for k, v in gpu.items()}
    RN.compare(op, inp, gpu, RN.run_oracle(orc, op, inp, 1e-5))


@pytest.mark.parametrize("op", ["ln", "rms", "add_rms"])
def test_absent_parameters(orc, op):
    inp = W.generic_rows(op, "bf16", 33, 768, seed=2)
    for k in ("gamma", "beta", "w"):
        inp.pop(k, None)
    _check(orc, op, inp)


@pytest.mark.parametrize("plan", [(nrm.PLAN_AUTO,), (nrm.PLAN_CTA, 128, 4), (nrm.PLAN_CTA, 256, 2),
                                  (nrm.PLAN_PERSIST,), (nrm.PLAN_WARP,), (nrm.PLAN_GENERIC, 256),
                                  (nrm.PLAN_CLUSTER, 128, 2, 0, 2), (nrm.PLAN_CLUSTER, 128, 1, 0, 4)],
                         ids=["auto", "cta128x4", "cta256x2", "persist", "warp", "generic",
                              "cluster128x2c2", "cluster128x1c4"])
@pytest.mark.parametrize("n", [1024, 2048, 4096])
def test_ln_small_spread_large_mean_f32(orc, n, plan):
    # binary32 rows with mean 1000 and spread 1e-3: the statistics must not
    # lose the spread to the mean's rounding (an error of one binary32 ulp of
    # 1000 in the mean would move y by 0.06)
    inp = W.generic_rows("ln", "f32", 16, n, seed=n + 5, scale=1e-3, shift=1000.0)
    nrm.force_plan(*plan)
    try:
        gpu = RN.run_gpu("ln", inp, 1e-12)
    except nrm.NrmError:
        pytest.skip("plan does not take this row length")
    RN.compare("ln", inp, gpu, RN.run_oracle(orc, "ln", inp, 1e-12))
    nrm.force_plan(nrm.PLAN_AUTO)


@pytest.mark.parametrize("dt", DTYPES)
def test_constant_rows_give_beta_exactly(dt):
    n = 4096
    inp = W.generic_rows("ln", dt, 8, n, seed=9)
    for i, c in enumerate([0.0, 1.0, 1000.0, -7.5, 3.25, 0.125, -1000.0, 42.0]):
        inp["x"][i] = c
    d = {k: v.cuda() for k, v in inp.items()}
    for plan in [(nrm.PLAN_AUTO, 0, 0), (nrm.PLAN_GENERIC, 256, 0), (nrm.PLAN_CTA, 1024, 1),
                 (nrm.PLAN_CLUSTER, 128, 4, 0, 2), (nrm.PLAN_CLUSTER, 128, 2, 0, 4)]:
        nrm.force_plan(*plan)
        y, mean, _ = nrm.ln_fwd(d["x"], d["gamma"], d["beta"], 1e-5)
        torch.cuda.synchronize()
        assert torch.equal(y.cpu(), inp["beta"].expand(8, n)), plan
        assert torch.equal(mean.cpu(), inp["x"][:, 0].float())


@pytest.mark.parametrize("plan", [(nrm.PLAN_CTA, 256, 2), (nrm.PLAN_CTA, 128, 4)],
                         ids=["cta256x2", "cta128x4"])
def test_zero_residual_equals_rms(plan):
    # on the same plan (same reduction order) a zero residual gives RMSNorm's
    # bits exactly
    inp = W.generic_rows("rms", "bf16", 64, 4096, seed=4)
    d = {k: v.cuda() for k, v in inp.items()}
    nrm.force_plan(*plan)
    y1, r1 = nrm.rms_fwd(d["x"], d["w"], 1e-6, want_stats=True)
    ro, y2, r2 = nrm.add_rms_fwd(d["x"], torch.zeros_like(d["x"]), d["w"], 1e-6, want_stats=True)
    assert torch.equal(ro, d["x"])
    assert torch.equal(y1, y2) and torch.equal(r1, r2)


def test_3d_input(orc):
    inp = W.generic_rows("rms", "f16", 4 * 24, 1024, seed=6)
    x3 = inp["x"].view(4, 24, 1024).cuda()
    y, rstd = nrm.rms_fwd(x3, inp["w"].cuda(), 1e-6, want_stats=True)
    assert y.shape == (4, 24, 1024) and rstd.shape == (4, 24)
    gpu = {"y": B.torch_to_np(y.view(96, 1024).cpu()), "rstd": rstd.view(96).cpu().numpy()}
    RN.compare("rms", inp, gpu, RN.run_oracle(orc, "rms", inp, 1e-6))


@pytest.mark.parametrize("op", ["ln", "add_rms"])
def test_guard_bands_untouched(op):
    rows, n, guard = 17, 1000, 256
    inp = W.generic_rows(op, "bf16", rows, n, seed=8)
    d = {k: v.cuda() for k, v in inp.items()}
    poison = -12345.0

    def guarded(shape, dtype):
        full = torch.full((int(np.prod(shape)) + 2 * guard,), poison, dtype=dtype, device="cuda")
        return full, full[guard:guard + int(np.prod(shape))].view(shape)

    fy, y = guarded((rows, n), torch.bfloat16)
    fs, s = guarded((rows,), torch.float32)
    if op == "ln":
        fm, m = guarded((rows,), torch.float32)
        nrm.ln_fwd(d["x"], d["gamma"], d["beta"], out=y, mean=m, rstd=s)
        fulls = [fy, fs, fm]
    else:
        fr, r = guarded((rows, n), torch.bfloat16)
        nrm.add_rms_fwd(d["x"], d["residual"], d["w"], residual_out=r, out=y, rstd=s)
        fulls = [fy, fs, fr]
    torch.cuda.synchronize()
    for f in fulls:
        assert torch.all(f[:guard] == poison) and torch.all(f[-guard:] == poison)


# ---- BatchNorm ------------------------------------------------------------
# automatic / streaming two kernels / cluster per channel / scalar two kernels /
# one-pass dataflow kernel
BN_PLANS = [nrm.PLAN_AUTO, nrm.PLAN_CTA, nrm.PLAN_TMA, nrm.PLAN_GENERIC, nrm.PLAN_PERSIST]
BN_IDS = ["auto", "stream", "cluster", "scalar", "flow"]


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("cs", [2, 4, 8, 16])
@pytest.mark.parametrize("shape", [(1, 1, 8, 8), (3, 5, 13, 12), (9, 6, 20, 20), (64, 3, 8, 8),
                                   (32, 4, 56, 56), (5, 2, 1, 4), (7, 3, 16, 24), (4, 2, 8, 257)])
def test_bn_cluster_sizes(orc, shape, cs, dtype):
    # the cluster plan at every cluster size; ranks beyond the batch hold no
    # planes.  16-bit planes arrive as one tensor copy per CTA where the shape
    # allows, the planes of a last CTA past the batch read as zeros; 8 x 257
    # planes have no box view (257 is prime) and keep the per-plane copies
    inp = W.make_inputs(W.BN_F32_32x64x56x56, shape=shape, dtype=dtype)
    nrm.force_plan(nrm.PLAN_TMA, 0, 0, cs, 0)
    gpu = RN.run_gpu("bn", inp, 1e-5, 0.1)
    # the cluster plan takes packed planes, at most 16 planes per CTA and two
    # buffers of at most 200 KB, or one of at most 220 KB; otherwise another
    # plan runs
    batch, hw = shape[0], shape[2] * shape[3]
    es = 4 if dtype == "f32" else 2
    while cs > 1 and cs > batch:
        cs //= 2
    ppc = -(-batch // cs)
    buf = -(-ppc * hw * es // 128) * 128
    fits = (hw * es) % 16 == 0 and ppc <= 16 and buf <= 220 * 1024
    assert (nrm.last_plan()[0] == nrm.PLAN_TMA) == fits
    RN.compare("bn", inp, gpu, RN.run_oracle(orc, "bn", inp, 1e-5, 0.1))


@pytest.mark.parametrize("shape,dtype,cs", [
    ((64, 20, 64, 64), "f32", 8), ((64, 20, 96, 96), "f32", 16), ((64, 9, 112, 112), "f32", 16),
    ((64, 20, 96, 96), "bf16", 0), ((64, 9, 112, 112), "bf16", 0), ((64, 20, 64, 64), "f16", 16)])
def test_bn_cluster_one_buffer(orc, shape, dtype, cs):
    # channels too large for two buffers per CTA: one buffer each, clusters of
    # up to 16 CTAs, more channels than resident clusters (each cluster takes
    # its channels one after another); the automatic size (cs 0) for 16-bit
    inp = W.make_inputs(W.BN_F32_32x64x56x56, shape=shape, dtype=dtype)
    nrm.force_plan(nrm.PLAN_TMA, 0, 0, cs, 0)
    gpu = RN.run_gpu("bn", inp, 1e-5, 0.1)
    assert nrm.last_plan()[0] == nrm.PLAN_TMA
    RN.compare("bn", inp, gpu, RN.run_oracle(orc, "bn", inp, 1e-5, 0.1))


@pytest.mark.parametrize("plan", BN_PLANS, ids=BN_IDS)
@pytest.mark.parametrize("shape", [(1, 1, 7, 7), (1, 3, 5, 5), (2, 4, 3, 3), (8, 16, 28, 28),
                                   (4, 8, 1, 1), (3, 5, 13, 11), (64, 3, 8, 8), (5, 7, 20, 20),
                                   (13, 2, 12, 12), (32, 4, 56, 56)])
def test_bn_shapes(orc, shape, plan):
    inp = W.make_inputs(W.BN_F32_32x64x56x56, shape=shape)
    nrm.force_plan(plan)
    gpu = RN.run_gpu("bn", inp, 1e-5, 0.1)
    ref = RN.run_oracle(orc, "bn", inp, 1e-5, 0.1)
    RN.compare("bn", inp, gpu, ref)


@pytest.mark.parametrize("plan", BN_PLANS, ids=BN_IDS)
def test_bn_large_mean_channel(orc, plan):
    inp = W.make_inputs(W.BN_F32_32x64x56x56, shape=(4, 3, 16, 16))
    inp["x"][:, 1] += 1000.0
    nrm.force_plan(plan)
    gpu = RN.run_gpu("bn", inp, 1e-5, 0.1)
    ref = RN.run_oracle(orc, "bn", inp, 1e-5, 0.1)
    RN.compare("bn", inp, gpu, ref)


def test_bn_plans_agree_and_repeat():
    inp = W.make_inputs(W.BN_F32_32x64x56x56, shape=(16, 8, 28, 28))
    outs = []
    plans = (nrm.PLAN_CTA, nrm.PLAN_CTA, nrm.PLAN_TMA, nrm.PLAN_TMA, nrm.PLAN_GENERIC,
             nrm.PLAN_PERSIST, nrm.PLAN_PERSIST, nrm.PLAN_TMA, nrm.PLAN_TMA)
    for i, plan in enumerate(plans):
        # the last two: the cluster plan with clusters of 8 CTAs (the first
        # two cluster runs take the automatic size)
        nrm.force_plan(plan, 0, 0, 8 if i >= 7 else 0, 0)
        outs.append(RN.run_gpu("bn", inp, 1e-5, 0.1))
        assert nrm.last_plan()[0] == plan
    for k in outs[0]:
        assert (outs[0][k] == outs[1][k]).all(), k  # bitwise repeatable
        assert (outs[2][k] == outs[3][k]).all(), k
        assert (outs[5][k] == outs[6][k]).all(), k
        assert (outs[7][k] == outs[8][k]).all(), k
        for o in (outs[2], outs[4], outs[5], outs[7]):
            assert np.max(np.abs(outs[0][k].astype(np.float64) - o[k])) <= 2e-5, k


def test_bn_without_optionals(orc):
    inp = W.make_inputs(W.BN_F32_32x64x56x56, shape=(2, 5, 6, 6))
    x = inp["x"].cuda()
    y, sm, sr = nrm.bn_fwd_train(x, None, None, None, None, 1e-5, 0.1)
    torch.cuda.synchronize()
    n = RN.to_np(inp)
    ref = orc.batchnorm_train(0, n["x"], eps=1e-5, wide=True)
    gy = y.cpu().numpy().reshape(ref["y_wide"].shape)
    assert np.max(np.abs(gy - ref["y_wide"])) <= 2e-5


@pytest.mark.parametrize("shape,dtype,cs", [
    ((16, 12, 28, 28), "f32", 0),    # two buffers, a bulk copy per plane
    ((16, 12, 28, 28), "bf16", 0),   # one tensor copy per CTA
    ((64, 20, 64, 64), "f32", 8),    # one buffer, channels one after another
    ((64, 20, 96, 96), "bf16", 0)])  # one buffer and tensor copies
def test_bn_cluster_wait_give_up_path(orc, shape, dtype, cs):
    # wait limit 0: every copy wait of the cluster plan gives up at once;
    # the kernel must raise the fault bit, keep every CTA in its cluster
    # barriers, drain its copies and return; the next call must be correct.
    inp = W.make_inputs(W.BN_F32_32x64x56x56, shape=shape, dtype=dtype)
    nrm.force_plan(nrm.PLAN_TMA, 0, 0, cs, 0)
    x = inp["x"].cuda()
    assert nrm.device_fault(clear=True) == 0
    old = nrm.set_wait_limit(0)
    try:
        nrm.bn_fwd_train(x, None, None, None, None, 1e-5, 0.1)
        bits = nrm.device_fault(clear=True)
    finally:
        nrm.set_wait_limit(old)
    assert bits == 1, bits
    gpu = RN.run_gpu("bn", inp, 1e-5, 0.1)
    RN.compare("bn", inp, gpu, RN.run_oracle(orc, "bn", inp, 1e-5, 0.1))
    assert nrm.device_fault(clear=True) == 0
