"""The oracle still reproduces its recorded outputs (tests/golden/oracle_regression.json)."""
import json
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))


def _arr(dt, hexes, shape):
    if dt == 0:
        return np.array([int(h, 16) for h in hexes], np.uint32).view(np.float32).reshape(shape)
    return np.array([int(h, 16) for h in hexes], np.uint16).reshape(shape)


def test_golden_regression(orc):
    data = json.load(open(os.path.join(HERE, "golden", "oracle_regression.json")))
    assert data["cases"]
    for c in data["cases"]:
        dt = c["dtype"]
        if c["op"] == "bn":
            shape = (c["batch"], c["c"], c["hw"])
            x = _arr(dt, c["x"], shape)
            g = _arr(dt, c["gamma"], (c["c"],))
            b = _arr(dt, c["beta"], (c["c"],))
            r = orc.batchnorm_train(dt, x, g, b, running_mean=[0.0] * c["c"],
                                    running_var=[1.0] * c["c"], eps=np.float32(c["eps"]),
                                    momentum=np.float32(c["momentum"]))
            assert np.array_equal(r["y"], _arr(dt, c["y"], shape))
            for k in ("save_mean", "save_rstd", "running_mean", "running_var"):
                assert np.array_equal(r[k], np.array(c[k]))
            continue
        if c["op"] == "bn_infer":
            shape = (c["batch"], c["c"], c["hw"])
            r = orc.batchnorm_infer(dt, _arr(dt, c["x"], shape), np.array(c["running_mean"]),
                                    np.array(c["running_var"]),
                                    _arr(dt, c["gamma"], (c["c"],)),
                                    _arr(dt, c["beta"], (c["c"],)), eps=np.float32(c["eps"]))
            assert np.array_equal(r["y"], _arr(dt, c["y"], shape))
            continue
        if c["op"] == "bn_bwd":
            shape = (c["batch"], c["c"], c["hw"])
            r = orc.batchnorm_backward(dt, _arr(dt, c["dy"], shape), _arr(dt, c["x"], shape),
                                       np.array(c["mean"]), np.array(c["rstd"]),
                                       _arr(dt, c["gamma"], (c["c"],)))
            assert np.array_equal(r["dx"], _arr(dt, c["dx"], shape))
            assert np.array_equal(r["dgamma"], np.array(c["dgamma"]))
            assert np.array_equal(r["dbeta"], np.array(c["dbeta"]))
            continue
        if c["op"] == "softmax":
            shape = (c["rows"], c["n"])
            r = orc.softmax(dt, _arr(dt, c["x"], shape))
            assert np.array_equal(r["y"], _arr(dt, c["y"], shape))
            assert np.array_equal(r["row_max"], np.array(c["row_max"]))
            assert np.array_equal(r["row_sum"], np.array(c["row_sum"]))
            continue
        shape = (c["rows"], c["n"])
        x = _arr(dt, c["x"], shape)
        if c["op"] == "ln":
            r = orc.layernorm(dt, x, _arr(dt, c["gamma"], (c["n"],)),
                              _arr(dt, c["beta"], (c["n"],)), eps=np.float32(c["eps"]))
            assert np.array_equal(r["mean"], np.array(c["mean"]))
        elif c["op"] == "rms":
            r = orc.rmsnorm(dt, x, _arr(dt, c["w"], (c["n"],)), eps=np.float32(c["eps"]))
        else:
            r = orc.add_rmsnorm(dt, x, _arr(dt, c["residual"], shape),
                                _arr(dt, c["w"], (c["n"],)), eps=np.float32(c["eps"]))
            assert np.array_equal(r["residual_out"], _arr(dt, c["residual_out"], shape))
        assert np.array_equal(r["y"], _arr(dt, c["y"], shape))
        assert np.array_equal(r["rstd"], np.array(c["rstd"]))
