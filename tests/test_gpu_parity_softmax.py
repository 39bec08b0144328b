"""Row softmax on the GPU against the CPU oracle: row lengths from 1 to 65536
(one pack, ragged tails, the register plan's limit and beyond it), every I/O
type, both plans, masked (-inf) entries, large logits, constant rows and
empty input."""
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


PLANS = [nrm.PLAN_AUTO, nrm.PLAN_GENERIC]
LENGTHS = [1, 2, 7, 8, 31, 64, 100, 1000, 1024, 2048, 4096, 4097, 8192, 16384, 32768, 65536]


def _inputs(dtype, rows, n, seed, scale=4.0, shift=0.0):
    return W.generic_rows("softmax", dtype, rows, n, seed, scale=scale, shift=shift)


@pytest.mark.parametrize("plan", PLANS, ids=["auto", "generic"])
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("n", LENGTHS)
def test_softmax_lengths(orc, n, dtype, plan):
    rows = 37 if n <= 4096 else 5
    inp = _inputs(dtype, rows, n, seed=n)
    nrm.force_plan(plan)
    gpu = RN.run_gpu("softmax", inp, 0.0)
    RN.compare("softmax", inp, gpu, RN.run_oracle(orc, "softmax", inp, 0.0))


@pytest.mark.parametrize("cfg", [(128, 1), (256, 1), (128, 4), (256, 2), (256, 4), (512, 4),
                                 (1024, 4)])
def test_softmax_forced_cta_shapes(orc, cfg):
    threads, packs = cfg
    n = 8 * min(threads * packs, 1024) - 8  # bf16 rows that leave some threads idle
    inp = _inputs("bf16", 9, n, seed=threads + packs)
    nrm.force_plan(nrm.PLAN_CTA, threads, packs)
    gpu = RN.run_gpu("softmax", inp, 0.0)
    RN.compare("softmax", inp, gpu, RN.run_oracle(orc, "softmax", inp, 0.0))


@pytest.mark.parametrize("plan", PLANS, ids=["auto", "generic"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_softmax_masked_large_and_constant(orc, dtype, plan):
    nrm.force_plan(plan)
    g = torch.Generator().manual_seed(3)
    inp = _inputs(dtype, 16, 2048, seed=11)
    x = inp["x"].float()
    mask = torch.rand(16, 2048, generator=g) < 0.3
    x[mask] = float("-inf")        # attention-style masking
    x[3] += 1000.0                 # large logits: the max keeps exp finite
    x[4] = 2.5                     # constant row: y = 1/N
    x[5, 1:] = float("-inf")       # one live entry: y = 1 there
    inp = {"x": x.to(inp["x"].dtype)}
    gpu = RN.run_gpu("softmax", inp, 0.0)
    RN.compare("softmax", inp, gpu, RN.run_oracle(orc, "softmax", inp, 0.0))
    assert np.all(RN.B.bits_to_f64(RN.B.dt_code(inp["x"].dtype), gpu["y"][5, 1:]) == 0.0)


@pytest.mark.parametrize("plan", [(nrm.PLAN_AUTO,), (nrm.PLAN_GENERIC,), (nrm.PLAN_CLUSTER, 128, 2, 0, 4)],
                         ids=["auto", "generic", "cluster"])
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_softmax_wide_logits_reach_subnormal_outputs(orc, dtype, plan):
    # logits spread over hundreds: many outputs fall below the smallest
    # normal (bfloat16 keeps subnormals down to 2^-133), which the fast
    # exponential path must neither flush early nor mis-round
    inp = _inputs(dtype, 24, 4096, seed=77, scale=45.0, shift=-5.0)
    nrm.force_plan(*plan)
    gpu = RN.run_gpu("softmax", inp, 0.0)
    RN.compare("softmax", inp, gpu, RN.run_oracle(orc, "softmax", inp, 0.0))
    y = RN.B.bits_to_f64(RN.B.dt_code(inp["x"].dtype), gpu["y"])
    if dtype == "bf16":  # the test does reach bfloat16 subnormal outputs
        assert np.any((y > 0) & (y < 2.0 ** -126))


def test_softmax_empty_and_repeatable():
    nrm.force_plan(nrm.PLAN_AUTO)
    x = torch.empty(0, 128, device="cuda")
    y, _, _ = nrm.softmax_fwd(x)
    assert y.shape == (0, 128)
    inp = W.make_inputs(W.SOFTMAX_BF16_4096x4096, shape=(512, 4096))
    a = RN.run_gpu("softmax", inp, 0.0)
    b = RN.run_gpu("softmax", inp, 0.0)
    for k in a:
        assert (a[k] == b[k]).all(), k
