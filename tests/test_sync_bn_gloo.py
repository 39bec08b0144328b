"""Synchronized BatchNorm's exchange on CPU ranks (gloo, world size 2).

Each rank holds half of a batch.  It computes its shard's per-channel
(count, mean, M2) with the oracle, exchanges them through the package's
exchange_parts (an all-gather in rank order), and combines the parts with
Chan's pairwise rule (written here from the LLM-ops page's "Welford combine"
formula).  The result must equal the oracle's statistics of the whole batch
(the reading of the BatchNorm page's §7.1: synchronized BatchNorm is
BatchNorm over the global batch), on every rank, bit for bit across ranks.
global_count must sum the local counts."""
import os
import sys

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HERE = os.path.dirname(os.path.abspath(__file__))


def _shard_stats(orc, x):
    """(count, mean, M2) per channel of one shard, from the oracle's training
    forward with eps = 0 (var = 1 / rstd^2)."""
    r = orc.batchnorm_train(0, x, eps=np.float32(0.0))
    cnt = x.shape[0] * x.shape[2]
    var = 1.0 / r["save_rstd"] ** 2
    return np.stack([np.full(x.shape[1], float(cnt)), r["save_mean"], var * cnt], axis=1)


def _chan(parts):
    n, mean, m2 = parts[0, :, 0].copy(), parts[0, :, 1].copy(), parts[0, :, 2].copy()
    for k in range(1, parts.shape[0]):
        nb, mb, m2b = parts[k, :, 0], parts[k, :, 1], parts[k, :, 2]
        tot = n + nb
        d = mb - mean
        mean = mean + d * nb / tot
        m2 = m2 + m2b + d * d * n * nb / tot
        n = tot
    return n, mean, m2


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, HERE)
    import oracle
    import row_wise_normalization_reduce_gb300 as nrm
    from row_wise_normalization_reduce_gb300 import workloads as W
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        orc = oracle.default()
        x = W.make_inputs(W.BN_F32_32x64x56x56, shape=(6, 5, 7, 9))["x"].numpy()
        x = x.reshape(6, 5, 63)
        shard = np.ascontiguousarray(x[3 * rank:3 * rank + 3])
        local = torch.from_numpy(_shard_stats(orc, shard))
        parts = nrm.exchange_parts(local).numpy()
        n, mean, m2 = _chan(parts)
        full = orc.batchnorm_train(0, x, eps=np.float32(0.0))
        out[rank] = {"parts": parts, "n": n, "mean": mean, "var": m2 / n,
                     "full_mean": full["save_mean"], "full_var": 1.0 / full["save_rstd"] ** 2,
                     "count": nrm.global_count(3 * 63, "cpu")}
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_sync_bn_exchange_gloo():
    port = 29600 + (os.getpid() % 1000)
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    a, b = res[0], res[1]
    assert np.array_equal(a["parts"], b["parts"])          # same parts, rank order
    assert np.array_equal(a["mean"], b["mean"]) and np.array_equal(a["var"], b["var"])
    assert np.all(a["n"] == 6 * 63) and a["count"] == b["count"] == 6 * 63
    assert np.allclose(a["mean"], a["full_mean"], rtol=1e-13, atol=1e-13)
    assert np.allclose(a["var"], a["full_var"], rtol=1e-12, atol=0)


def test_single_process_exchange_is_identity():
    sys.path.insert(0, ROOT)
    import row_wise_normalization_reduce_gb300 as nrm
    t = torch.arange(12, dtype=torch.float64).reshape(4, 3)
    p = nrm.exchange_parts(t)
    assert p.shape == (1, 4, 3) and torch.equal(p[0], t)
    assert nrm.global_count(17, "cpu") == 17
