"""Run the same seeded inputs through the CUDA library (via the C ABI binding)
and through the CPU oracle, and compare them with the stated tolerances."""
import numpy as np
import torch

import bits as B
import tolerance as T


def to_np(d):
    return {k: (None if v is None else B.torch_to_np(v)) for k, v in d.items()}


def run_gpu(op, inp, eps, momentum=0.1, device="cuda", residual_inplace=False):
    import row_wise_normalization_reduce_gb300 as nrm
    d = {k: (None if v is None else v.to(device)) for k, v in inp.items()}
    out = {}
    if op == "ln":
        y, mean, rstd = nrm.ln_fwd(d["x"], d.get("gamma"), d.get("beta"), eps)
        out = {"y": y, "mean": mean, "rstd": rstd}
    elif op == "rms":
        y, rstd = nrm.rms_fwd(d["x"], d.get("w"), eps, want_stats=True)
        out = {"y": y, "rstd": rstd}
    elif op == "add_rms":
        if residual_inplace:
            res = d["residual"].clone()
            ro, y, rstd = nrm.add_rms_fwd(d["x"], res, d.get("w"), eps, residual_out=res,
                                          want_stats=True)
            assert ro.data_ptr() == res.data_ptr()
        else:
            ro, y, rstd = nrm.add_rms_fwd(d["x"], d["residual"], d.get("w"), eps, want_stats=True)
        out = {"residual_out": ro, "y": y, "rstd": rstd}
    elif op == "bn":
        rm = d["running_mean"].clone()
        rv = d["running_var"].clone()
        y, sm, sr = nrm.bn_fwd_train(d["x"], d.get("gamma"), d.get("beta"), rm, rv, eps, momentum)
        out = {"y": y, "save_mean": sm, "save_rstd": sr, "running_mean": rm, "running_var": rv}
    elif op == "bn_infer":
        y = nrm.bn_fwd_infer(d["x"], d["running_mean"], d["running_var"], d.get("gamma"),
                             d.get("beta"), eps)
        out = {"y": y}
    elif op == "bn_bwd":
        dx, dg, db = nrm.bn_bwd(d["dy"], d["x"], d["save_mean"], d["save_rstd"], d.get("gamma"))
        out = {"dx": dx, "dgamma": dg, "dbeta": db}
    elif op == "softmax":
        y, m, sm = nrm.softmax_fwd(d["x"], want_stats=True)
        out = {"y": y, "row_max": m, "row_sum": sm}
    torch.cuda.synchronize()
    return {k: B.torch_to_np(v.cpu()) for k, v in out.items()}


def run_oracle(orc, op, inp, eps, momentum=0.1):
    n = to_np(inp)
    dt = B.dt_code(inp["x"].dtype)
    if op == "ln":
        return orc.layernorm(dt, n["x"], n.get("gamma"), n.get("beta"), eps=eps, wide=True)
    if op == "rms":
        return orc.rmsnorm(dt, n["x"], n.get("w"), eps=eps, wide=True)
    if op == "add_rms":
        return orc.add_rmsnorm(dt, n["x"], n["residual"], n.get("w"), eps=eps, wide=True)
    if op == "bn":
        x = n["x"]
        r = orc.batchnorm_train(dt, x, n.get("gamma"), n.get("beta"),
                                n["running_mean"].astype(np.float64),
                                n["running_var"].astype(np.float64), eps=eps, momentum=momentum,
                                wide=True)
        r["y"] = r["y"].reshape(x.shape)
        r["y_wide"] = r["y_wide"].reshape(x.shape)
        return r
    if op == "bn_infer":
        x = n["x"]
        r = orc.batchnorm_infer(dt, x, n["running_mean"], n["running_var"], n.get("gamma"),
                                n.get("beta"), eps=eps, wide=True)
        r["y"] = r["y"].reshape(x.shape)
        r["y_wide"] = r["y_wide"].reshape(x.shape)
        return r
    if op == "bn_bwd":
        x = n["x"]
        r = orc.batchnorm_backward(dt, n["dy"], x, n["save_mean"].astype(np.float64),
                                   n["save_rstd"].astype(np.float64), n.get("gamma"), wide=True)
        r["dx"] = r["dx"].reshape(x.shape)
        r["dx_wide"] = r["dx_wide"].reshape(x.shape)
        return r
    if op == "softmax":
        return orc.softmax(dt, n["x"], wide=True)
    raise ValueError(op)


def select_channels(op, inp, chans):
    """The inputs of BatchNorm channels `chans` only (channels are independent,
    so the oracle on them gives the exact reference for those channels)."""
    out = {}
    for k, v in inp.items():
        if v is None:
            out[k] = None
        elif v.dim() >= 2:
            out[k] = v[:, chans].contiguous()
        else:
            out[k] = v[chans].contiguous()
    return out


def slice_gpu_channels(gpu, chans):
    return {k: (v[:, chans] if v.ndim >= 2 else v[chans]) for k, v in gpu.items()}


def compare(op, inp, gpu, ref):
    """Assert parity; return measured errors."""
    dt = B.dt_code(inp["x"].dtype)
    n = to_np(inp)
    rep = {}
    if op == "ln":
        scale = T.ln_affine_scale(dt, n["x"], ref["mean"], ref["rstd"], n.get("gamma"),
                                  n.get("beta"))
        rep["y"] = T.check_y(dt, gpu["y"], ref["y"], ref["y_wide"], scale)
        var = 1.0 / ref["rstd"] ** 2
        rep["mean"] = T.check_stat(gpu["mean"], ref["mean"], "mean",
                                   scale=np.abs(ref["mean"]) + np.sqrt(var))
        rep["rstd"] = T.check_stat(gpu["rstd"], ref["rstd"], "rstd")
    elif op in ("rms", "add_rms"):
        if op == "add_rms":
            assert np.array_equal(gpu["residual_out"], ref["residual_out"]), "residual_out not bit-exact"
            rep["residual_out"] = "bit-exact"
        rep["y"] = T.check_y(dt, gpu["y"], ref["y"], ref["y_wide"], None)
        rep["rstd"] = T.check_stat(gpu["rstd"], ref["rstd"], "rstd")
    elif op == "bn":
        c = n["x"].shape[1]
        view = (1, c) + (1,) * (n["x"].ndim - 2)
        x64 = B.bits_to_f64(dt, n["x"])
        t = (x64 - ref["save_mean"].reshape(view)) * ref["save_rstd"].reshape(view)
        g = 1.0 if n.get("gamma") is None else B.bits_to_f64(dt, n["gamma"]).reshape(view)
        b = 0.0 if n.get("beta") is None else B.bits_to_f64(dt, n["beta"]).reshape(view)
        rep["y"] = T.check_y(dt, gpu["y"], ref["y"], ref["y_wide"],
                             np.abs(t * g) + np.abs(b) + np.abs(g))
        var = 1.0 / ref["save_rstd"] ** 2 - 0.0
        rep["save_mean"] = T.check_stat(gpu["save_mean"], ref["save_mean"], "save_mean",
                                        scale=np.abs(ref["save_mean"]) + np.sqrt(var))
        rep["save_rstd"] = T.check_stat(gpu["save_rstd"], ref["save_rstd"], "save_rstd")
        rep["running_mean"] = T.check_stat(gpu["running_mean"], ref["running_mean"],
                                           "running_mean",
                                           scale=np.abs(ref["running_mean"]) + np.sqrt(var))
        rep["running_var"] = T.check_stat(gpu["running_var"], ref["running_var"], "running_var")
    elif op == "bn_infer":
        c = n["x"].shape[1]
        view = (1, c) + (1,) * (n["x"].ndim - 2)
        x64 = B.bits_to_f64(dt, n["x"])
        rm = n["running_mean"].astype(np.float64).reshape(view)
        rv = n["running_var"].astype(np.float64).reshape(view)
        t = (x64 - rm) / np.sqrt(rv)  # eps left out: a slightly larger bound
        g = 1.0 if n.get("gamma") is None else B.bits_to_f64(dt, n["gamma"]).reshape(view)
        b = 0.0 if n.get("beta") is None else B.bits_to_f64(dt, n["beta"]).reshape(view)
        rep["y"] = T.check_y(dt, gpu["y"], ref["y"], ref["y_wide"],
                             np.abs(t * g) + np.abs(b) + np.abs(g))
    elif op == "bn_bwd":
        c = n["x"].shape[1]
        view = (1, c) + (1,) * (n["x"].ndim - 2)
        axes = (0,) + tuple(range(2, n["x"].ndim))
        x64 = B.bits_to_f64(dt, n["x"])
        dy = B.bits_to_f64(dt, n["dy"])
        rstd = n["save_rstd"].astype(np.float64).reshape(view)
        xh = (x64 - n["save_mean"].astype(np.float64).reshape(view)) * rstd
        g = 1.0 if n.get("gamma") is None else B.bits_to_f64(dt, n["gamma"]).reshape(view)
        cnt = dy.size // c
        s1 = np.abs(dy).sum(axis=axes)
        s2 = np.abs(dy * xh).sum(axis=axes)
        scale = np.abs(g) * rstd * (np.abs(dy) + (np.abs(ref["dbeta"]) + s1).reshape(view) / cnt
                                   + np.abs(xh) * (np.abs(ref["dgamma"]) + s2).reshape(view) / cnt)
        rep["dx"] = T.check_scaled(dt, gpu["dx"], ref["dx"], ref["dx_wide"], scale, T.BWD_REL,
                                   "dx")
        rep["dbeta"] = T.check_stat(gpu["dbeta"], ref["dbeta"], "dbeta", scale=s1)
        rep["dgamma"] = T.check_stat(gpu["dgamma"], ref["dgamma"], "dgamma", scale=s2)
    elif op == "softmax":
        rep["y"] = T.check_softmax(dt, gpu["y"], ref["y"], ref["y_wide"])
        # the max of stored values is exact in any precision
        assert np.array_equal(gpu["row_max"].astype(np.float64), ref["row_max"]), "row_max"
        rep["row_sum"] = T.check_stat(gpu["row_sum"], ref["row_sum"], "row_sum",
                                      scale=np.abs(ref["row_sum"]) * (T.SOFTMAX_REL / T.STAT_REL))
    return rep
