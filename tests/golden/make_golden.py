"""Write tests/golden/oracle_regression.json from the CPU oracle alone.

The pages print no input/output values for a worked example, so this fixture
is a regression record of the oracle on small, explicitly defined inputs
(integer patterns, no random generator, identical on every platform).  It is
written only by this script, which calls nothing but ``oracle``.

Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
import oracle  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_regression.json")


def pattern(rows, n, mul, mod, off, scale):
    i = np.arange(rows * n).reshape(rows, n)
    return ((i * mul + off) % mod - mod // 2) / scale


def storage(dt, v):
    orc = oracle.default()
    v = np.asarray(v, np.float64)
    if dt == 0:
        return v.astype(np.float32)
    enc = orc.double_to_f16 if dt == 1 else orc.double_to_bf16
    return np.array([enc(float(t)) for t in v.ravel()], np.uint16).reshape(v.shape)


def hexs(a):
    a = np.asarray(a)
    if a.dtype == np.float32:
        return [format(int(t), "08x") for t in a.view(np.uint32).ravel()]
    return [format(int(t), "04x") for t in a.ravel()]


def cases():
    orc = oracle.default()
    out = []
    for dt, rows, n in ((0, 3, 20), (2, 2, 33), (1, 2, 16)):
        x = storage(dt, pattern(rows, n, 37, 29, 5, 8.0) + 3.0)
        g = storage(dt, 1.0 + pattern(1, n, 5, 9, 1, 16.0)[0])
        b = storage(dt, pattern(1, n, 7, 11, 2, 32.0)[0])
        r = orc.layernorm(dt, x, g, b, eps=np.float32(1e-5))
        out.append({"op": "ln", "dtype": dt, "rows": rows, "n": n, "eps": 1e-5,
                    "x": hexs(x), "gamma": hexs(g), "beta": hexs(b),
                    "y": hexs(r["y"]), "mean": r["mean"].tolist(), "rstd": r["rstd"].tolist()})
    for dt, rows, n in ((1, 2, 24), (2, 2, 17)):
        x = storage(dt, pattern(rows, n, 13, 31, 3, 4.0))
        w = storage(dt, 1.0 + pattern(1, n, 3, 7, 0, 32.0)[0])
        r = orc.rmsnorm(dt, x, w, eps=np.float32(1e-6))
        out.append({"op": "rms", "dtype": dt, "rows": rows, "n": n, "eps": 1e-6,
                    "x": hexs(x), "w": hexs(w), "y": hexs(r["y"]), "rstd": r["rstd"].tolist()})
    for dt, rows, n in ((2, 3, 16), (1, 2, 12)):
        x = storage(dt, pattern(rows, n, 11, 23, 1, 4.0))
        res = storage(dt, pattern(rows, n, 17, 19, 4, 3.0))
        w = storage(dt, 1.0 + pattern(1, n, 3, 5, 1, 16.0)[0])
        r = orc.add_rmsnorm(dt, x, res, w, eps=np.float32(1e-6))
        out.append({"op": "add_rms", "dtype": dt, "rows": rows, "n": n, "eps": 1e-6,
                    "x": hexs(x), "residual": hexs(res), "w": hexs(w),
                    "residual_out": hexs(r["residual_out"]), "y": hexs(r["y"]),
                    "rstd": r["rstd"].tolist()})
    batch, c, hw = 2, 3, 5
    x = storage(0, pattern(batch * c, hw, 7, 13, 2, 2.0).reshape(batch, c, hw) + 1.0)
    g = storage(0, [1.0, 0.5, 1.25])
    b = storage(0, [0.0, 0.25, -0.5])
    r = orc.batchnorm_train(0, x, g, b, running_mean=[0.0] * c, running_var=[1.0] * c,
                            eps=np.float32(1e-5), momentum=np.float32(0.1))
    out.append({"op": "bn", "dtype": 0, "batch": batch, "c": c, "hw": hw, "eps": 1e-5,
                "momentum": 0.1, "x": hexs(x), "gamma": hexs(g), "beta": hexs(b),
                "y": hexs(r["y"]), "save_mean": r["save_mean"].tolist(),
                "save_rstd": r["save_rstd"].tolist(),
                "running_mean": r["running_mean"].tolist(),
                "running_var": r["running_var"].tolist()})
    for dt in (0, 2):
        x = storage(dt, pattern(batch * c, hw, 5, 17, 3, 4.0).reshape(batch, c, hw))
        g = storage(dt, [1.0, 0.75, 1.5])
        b = storage(dt, [0.5, 0.0, -0.25])
        rm = np.array([0.25, -1.0, 2.0], np.float32)
        rv = np.array([1.5, 0.5, 4.0], np.float32)
        r = orc.batchnorm_infer(dt, x, rm, rv, g, b, eps=np.float32(1e-5))
        out.append({"op": "bn_infer", "dtype": dt, "batch": batch, "c": c, "hw": hw,
                    "eps": 1e-5, "x": hexs(x), "gamma": hexs(g), "beta": hexs(b),
                    "running_mean": rm.tolist(), "running_var": rv.tolist(), "y": hexs(r["y"])})
    for dt in (0, 1):
        x = storage(dt, pattern(batch * c, hw, 7, 13, 2, 2.0).reshape(batch, c, hw) + 1.0)
        dy = storage(dt, pattern(batch * c, hw, 11, 19, 4, 8.0).reshape(batch, c, hw))
        g = storage(dt, [1.0, 0.5, 1.25])
        mean = [1.0, 0.75, 1.25]
        rstd = [0.5, 0.625, 0.375]
        r = orc.batchnorm_backward(dt, dy, x, mean, rstd, g)
        out.append({"op": "bn_bwd", "dtype": dt, "batch": batch, "c": c, "hw": hw,
                    "x": hexs(x), "dy": hexs(dy), "gamma": hexs(g), "mean": mean,
                    "rstd": rstd, "dx": hexs(r["dx"]), "dgamma": r["dgamma"].tolist(),
                    "dbeta": r["dbeta"].tolist()})
    for dt, rows, n in ((0, 3, 19), (2, 2, 24), (1, 2, 9)):
        x = storage(dt, pattern(rows, n, 23, 41, 6, 4.0))
        r = orc.softmax(dt, x)
        out.append({"op": "softmax", "dtype": dt, "rows": rows, "n": n, "x": hexs(x),
                    "y": hexs(r["y"]), "row_max": r["row_max"].tolist(),
                    "row_sum": r["row_sum"].tolist()})
    return out


if __name__ == "__main__":
    with open(OUT, "w") as f:
        json.dump({"source": "written by tests/golden/make_golden.py from the CPU oracle",
                   "cases": cases()}, f, indent=0)
    print("wrote", OUT)
