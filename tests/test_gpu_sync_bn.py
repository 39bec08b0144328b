"""Synchronized BatchNorm's kernels on one GPU: the batch is split into parts
as separate processes would hold it; each part's partial statistics (sums
for the backward) are computed, the arrays stacked in rank order (what the
all-gather produces) and each part normalized (differentiated) with them.
Every part's outputs must match the oracle on the whole batch.  No kernel
waits on another: the parts run one after another on one stream."""
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


SPLITS = [(4, 8, 14, 14, [2, 2]), (6, 3, 9, 11, [1, 2, 3]), (8, 16, 28, 28, [3, 5]),
          (2, 4, 5, 5, [1, 1])]


# partial statistics: the cluster plan in statistics-only mode (automatic, for
# packed planes) or the streaming units and a binary64 fold (forced)
@pytest.mark.parametrize("plan", [nrm.PLAN_AUTO, nrm.PLAN_CTA], ids=["auto", "stream"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("split", SPLITS, ids=lambda s: "x".join(map(str, s[:4])) + "_" +
                         "-".join(map(str, s[4])))
def test_sync_bn_forward_parts_match_whole_batch(orc, split, dtype, plan):
    shape, sizes = tuple(split[:4]), split[4]
    inp = W.make_inputs(W.BN_F32_32x64x56x56, shape=shape, dtype=dtype)
    x = inp["x"].cuda()
    g, b = inp["gamma"].cuda(), inp["beta"].cuda()
    shards = torch.split(x, sizes, dim=0)
    nrm.force_plan(plan)
    try:
        parts = torch.stack([nrm.bn_fwd_partial_stats(s) for s in shards])
    finally:
        nrm.force_plan(nrm.PLAN_AUTO)
    ys, rms, rvs = [], [], []
    for s in shards:
        rm = inp["running_mean"].cuda()
        rv = inp["running_var"].cuda()
        y, sm, sr = nrm.bn_fwd_apply_stats(s, parts, g, b, rm, rv, 1e-5, 0.1)
        ys.append(y)
        rms.append(rm)
        rvs.append(rv)
    torch.cuda.synchronize()
    gpu = {"y": RN.B.torch_to_np(torch.cat(ys).cpu()), "save_mean": sm.cpu().numpy(),
           "save_rstd": sr.cpu().numpy(), "running_mean": rms[0].cpu().numpy(),
           "running_var": rvs[0].cpu().numpy()}
    for other in rms[1:]:
        assert torch.equal(other, rms[0])
    RN.compare("bn", inp, gpu, RN.run_oracle(orc, "bn", inp, 1e-5, 0.1))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("split", SPLITS, ids=lambda s: "x".join(map(str, s[:4])) + "_" +
                         "-".join(map(str, s[4])))
def test_sync_bn_backward_parts_match_whole_batch(orc, split, dtype):
    shape, sizes = tuple(split[:4]), split[4]
    inp = W.make_inputs(W.BN_BWD_F32_32x64x56x56, shape=shape, dtype=dtype)
    x, dy = inp["x"].cuda(), inp["dy"].cuda()
    sm, sr, g = inp["save_mean"].cuda(), inp["save_rstd"].cuda(), inp["gamma"].cuda()
    xs, dys = torch.split(x, sizes, dim=0), torch.split(dy, sizes, dim=0)
    parts = torch.stack([nrm.bn_bwd_partial_sums(d, s, sm, sr) for d, s in zip(dys, xs)])
    count = x.numel() // x.shape[1]
    outs = [nrm.bn_bwd_apply_sums(d, s, sm, sr, parts, count, g) for d, s in zip(dys, xs)]
    torch.cuda.synchronize()
    gpu = {"dx": RN.B.torch_to_np(torch.cat([o[0] for o in outs]).cpu()),
           "dgamma": outs[0][1].cpu().numpy(), "dbeta": outs[0][2].cpu().numpy()}
    RN.compare("bn_bwd", inp, gpu, RN.run_oracle(orc, "bn_bwd", inp, 1e-5))


def test_sync_bn_single_process_matches_bn_fwd_train():
    inp = W.make_inputs(W.BN_F32_32x64x56x56, shape=(8, 16, 28, 28))
    x = inp["x"].cuda()
    y1, m1, r1 = nrm.sync_bn_fwd_train(x, inp["gamma"].cuda(), inp["beta"].cuda())
    y2, m2, r2 = nrm.bn_fwd_train(x, inp["gamma"].cuda(), inp["beta"].cuda())
    torch.cuda.synchronize()
    assert torch.max(torch.abs(y1 - y2)).item() <= 2e-5
    assert torch.allclose(m1, m2, rtol=1e-5, atol=1e-5) and torch.allclose(r1, r2, rtol=1e-5)
