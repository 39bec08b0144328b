"""Pins for the CPU oracle: facts fixed by the pages' formulas and by mathematics,
checked without trusting the oracle's own code.

Each pin is a function of an ``oracle.Oracle`` (so the same pins can be run
against deliberately broken oracle builds, see test_oracle_mutants.py) and
raises AssertionError when the oracle disagrees with:
  * exact rational arithmetic (fractions / 60-digit decimals) on tiny inputs,
  * closed forms (arithmetic sequences, constant rows, +-1 patterns),
  * invariants (shift invariance, standardized moments, scaling),
  * an independent algorithm (the Welford recurrence of the LLM-ops page,
    smarter.xin, "Welford recurrence" section),
  * independent library conversions (numpy float16, torch bfloat16/float32).

The pages print no input/output values for a worked example, so no pin quotes
page numbers; every expected value is derived here from the definitions.
"""
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np

import bits as B

getcontext().prec = 60
F32, F16, BF16 = 0, 1, 2


# --------------------------------------------------------------------------
# helpers (exact arithmetic; nothing here calls the oracle)
# --------------------------------------------------------------------------
def _enc(dt, values):
    """Encode exactly-representable doubles into the oracle's storage arrays."""
    v = np.asarray(values, np.float64)
    if dt == F32:
        out = v.astype(np.float32)
        assert np.array_equal(out.astype(np.float64), v)
        return out
    if dt == F16:
        out = B.f64_to_bits_numpy_f16(v)
        assert np.array_equal(B.f16_bits_to_f64(out), v)
        return out
    out = B.f32_to_bits_torch_bf16(v.astype(np.float32))
    assert np.array_equal(B.bf16_bits_to_f64(out), v)
    return out


def _dec(x):
    return Decimal(Fraction(float(x)).numerator) / Decimal(Fraction(float(x)).denominator)


def _exact_ln_row(xs, gs, bs, eps):
    """Exact mean/var (Fractions) and 60-digit y for one LayerNorm row."""
    fx = [Fraction(float(v)) for v in xs]
    n = len(fx)
    mean = sum(fx) / n
    var = sum((v - mean) ** 2 for v in fx) / n
    den = (Decimal(var.numerator) / Decimal(var.denominator) + _dec(eps)).sqrt()
    dmean = Decimal(mean.numerator) / Decimal(mean.denominator)
    ys = [(_dec(v) - dmean) / den * _dec(g) + _dec(b) for v, g, b in zip(xs, gs, bs)]
    return mean, var, Decimal(1) / den, ys


def _close(a, b, rel, absol=0.0):
    a = float(a)
    b = float(b)
    assert abs(a - b) <= absol + rel * abs(b), (a, b)


# --------------------------------------------------------------------------
# IEEE storage conversions
# --------------------------------------------------------------------------
def pin_f16_decode_exhaustive(orc):
    allbits = np.arange(65536, dtype=np.uint16)
    ref = B.f16_bits_to_f64(allbits)
    got = np.array([orc.f16_to_double(int(b)) for b in allbits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def pin_bf16_decode_exhaustive(orc):
    allbits = np.arange(65536, dtype=np.uint16)
    ref = B.bf16_bits_to_f64(allbits)
    got = np.array([orc.bf16_to_double(int(b)) for b in allbits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def pin_roundtrip_exhaustive(orc):
    for dec, enc, to64 in ((orc.f16_to_double, orc.double_to_f16, B.f16_bits_to_f64),
                           (orc.bf16_to_double, orc.double_to_bf16, B.bf16_bits_to_f64)):
        for b in range(65536):
            v = to64(np.uint16(b))
            e = enc(float(v))
            if np.isnan(v):
                assert np.isnan(to64(np.uint16(e))) and (e >> 15) == (b >> 15)
            else:
                assert e == b, (hex(b), hex(e))


def pin_f16_encode_matches_numpy(orc):
    rng = np.random.default_rng(11)
    mags = np.concatenate([
        rng.uniform(0, 1, 3000) * 2.0 ** rng.integers(-30, 17, 3000),  # incl. subnormal/overflow
        rng.standard_normal(2000),
        np.array([65504.0, 65519.99, 65520.0, 65535.0, 2.0 ** -24, 2.0 ** -25,
                  3 * 2.0 ** -25, 2.0 ** -26, 6.1e-5, 1e-9, 0.0])])
    vals = np.concatenate([mags, -mags])
    ref = B.f64_to_bits_numpy_f16(vals)
    got = np.array([orc.double_to_f16(float(v)) for v in vals], np.uint16)
    bad = np.nonzero(ref != got)[0]
    assert bad.size == 0, [(vals[i], hex(ref[i]), hex(got[i])) for i in bad[:5]]


def pin_bf16_encode_matches_torch(orc):
    rng = np.random.default_rng(12)
    f = np.concatenate([
        (rng.uniform(-1, 1, 4000) * 2.0 ** rng.integers(-140, 128, 4000)).astype(np.float32),
        rng.standard_normal(2000).astype(np.float32),
        np.array([3.3895314e38, 3.4e38, 1e-40, 9.2e-41, 1.0 + 2.0 ** -8], np.float32)])
    f = f[np.isfinite(f)]
    ref = B.f32_to_bits_torch_bf16(f)
    got = np.array([orc.double_to_bf16(float(v)) for v in f], np.uint16)
    bad = np.nonzero(ref != got)[0]
    assert bad.size == 0, [(f[i], hex(ref[i]), hex(got[i])) for i in bad[:5]]


def pin_ties_and_edges(orc):
    # bfloat16: 1 + 2^-8 is halfway between 1 and 1 + 2^-7 -> even (1.0)
    assert orc.double_to_bf16(1.0 + 2.0 ** -8) == 0x3F80
    assert orc.double_to_bf16(1.0 + 3 * 2.0 ** -8) == 0x3F82
    assert orc.double_to_bf16(-(1.0 + 2.0 ** -8)) == 0xBF80
    assert orc.double_to_bf16(1.0 + 2.0 ** -8 + 2.0 ** -30) == 0x3F81
    # binary16
    assert orc.double_to_f16(1.0 + 2.0 ** -11) == 0x3C00
    assert orc.double_to_f16(1.0 + 3 * 2.0 ** -11) == 0x3C02
    assert orc.double_to_f16(65520.0) == 0x7C00          # tie at the top -> inf
    assert orc.double_to_f16(65519.0) == 0x7BFF
    assert orc.double_to_f16(2.0 ** -25) == 0x0000       # half the smallest subnormal -> 0
    assert orc.double_to_f16(3 * 2.0 ** -25) == 0x0002   # tie -> even subnormal
    assert orc.double_to_f16(2.0 ** -14 - 2.0 ** -25) == 0x0400  # rounds up into the normals
    assert orc.double_to_f16(-0.0) == 0x8000
    assert orc.double_to_f16(float("inf")) == 0x7C00
    assert orc.double_to_bf16(float("-inf")) == 0xFF80
    # overflow well past the largest finite value
    assert orc.double_to_f16(70000.0) == 0x7C00
    assert orc.double_to_f16(-1e300) == 0xFC00
    assert orc.double_to_bf16(3.5e38) == 0x7F80
    assert orc.double_to_bf16(1e300) == 0x7F80
    # binary32 (C cast) against numpy
    for v in (1.0 + 2.0 ** -24, 1.0 + 3 * 2.0 ** -24, 0.1, 1e-45, 3.5e38, 1e39):
        with np.errstate(over="ignore"):  # 1e39 rounds to infinity on both sides
            assert np.float32(orc.double_to_f32(v)) == np.float64(v).astype(np.float32)


# --------------------------------------------------------------------------
# LayerNorm
# --------------------------------------------------------------------------
def pin_ln_exact_tiny(orc):
    rng = np.random.default_rng(21)
    for dt in (F32, F16, BF16):
        for n in (1, 2, 3, 5, 8):
            xs = rng.integers(-40, 41, size=(3, n)).astype(np.float64) / 4.0
            gs = rng.integers(-8, 9, size=n).astype(np.float64) / 8.0
            bs = rng.integers(-8, 9, size=n).astype(np.float64) / 16.0
            eps = np.float32(1e-5)
            r = orc.layernorm(dt, _enc(dt, xs), _enc(dt, gs), _enc(dt, bs), eps=eps, wide=True)
            for i in range(3):
                mean, var, rstd, ys = _exact_ln_row(xs[i], gs, bs, eps)
                _close(r["mean"][i], mean, 1e-15, 1e-15)
                _close(r["rstd"][i], rstd, 1e-14)
                for j in range(n):
                    _close(r["y_wide"][i, j], ys[j], 1e-13, 1e-13)


def pin_ln_arithmetic_sequence(orc):
    for a, d, n in ((3.0, 0.5, 1024), (-7.0, 2.0, 129), (1000.0, 0.25, 4096), (0.0, 1.0, 2)):
        row = a + d * np.arange(n)
        r = orc.layernorm(F32, _enc(F32, row[None, :]), eps=np.float32(0.0))
        mean = a + d * (n - 1) / 2.0
        var = d * d * (n * n - 1) / 12.0
        _close(r["mean"][0], mean, 1e-15, 1e-15)
        _close(1.0 / r["rstd"][0] ** 2, var, 1e-12)


def pin_ln_welford_matches(orc):
    # The Welford recurrence (delta = x_k - mu_{k-1}; mu_k = mu_{k-1} + delta/k;
    # M2_k = M2_{k-1} + delta*(x_k - mu_k); var = M2_n/n), run in Python doubles.
    rng = np.random.default_rng(22)
    xs = (rng.standard_normal((6, 7)) * 3 + 2).astype(np.float32)
    eps = np.float32(1e-5)
    r = orc.layernorm(F32, xs, eps=eps)
    for i in range(xs.shape[0]):
        mu, m2 = 0.0, 0.0
        for k, v in enumerate(xs[i].astype(np.float64), start=1):
            delta = v - mu
            mu += delta / k
            m2 += delta * (v - mu)
        _close(r["mean"][i], mu, 1e-13, 1e-13)
        _close(r["rstd"][i], 1.0 / np.sqrt(m2 / xs.shape[1] + float(eps)), 1e-12)


def pin_ln_constant_rows_give_beta(orc):
    rng = np.random.default_rng(23)
    for dt in (F32, F16, BF16):
        n = 67
        beta = _enc(dt, rng.integers(-64, 65, n) / 64.0)
        gamma = _enc(dt, 1.0 + rng.integers(-8, 9, n) / 16.0)
        for c in (0.0, 1.5, 1000.0, -7.5):
            x = _enc(dt, np.full((2, n), c))
            r = orc.layernorm(dt, x, gamma, beta, eps=np.float32(1e-5))
            assert np.array_equal(r["y"], np.broadcast_to(beta, (2, n)))
            assert np.all(r["mean"] == c)


def pin_ln_standardized_moments(orc):
    rng = np.random.default_rng(24)
    x = (rng.standard_normal((4, 513)) * 2.5 + 3.0).astype(np.float32)
    eps = np.float32(1e-5)
    r = orc.layernorm(F32, x, eps=eps, wide=True)
    y = r["y_wide"]
    for i in range(4):
        xv = x[i].astype(np.float64)
        var = np.mean((xv - xv.mean()) ** 2)
        assert abs(y[i].mean()) <= 1e-12
        _close(np.mean(y[i] ** 2), var / (var + float(eps)), 1e-12)


def pin_ln_shift_invariance(orc):
    rng = np.random.default_rng(25)
    base = rng.integers(-2048, 2048, size=(3, 300)) / 256.0
    g = _enc(F32, 1.0 + rng.integers(-8, 9, 300) / 16.0)
    b = _enc(F32, rng.integers(-8, 9, 300) / 16.0)
    ref = orc.layernorm(F32, _enc(F32, base), g, b, wide=True)["y_wide"]
    for c in (1000.0, -7.5):
        got = orc.layernorm(F32, _enc(F32, base + c), g, b, wide=True)["y_wide"]
        assert np.max(np.abs(got - ref)) <= 1e-12


def pin_ln_affine_roles(orc):
    # gamma multiplies element i, beta adds to element i (non-symmetric vectors so
    # a reversed or shifted index shows up).
    rng = np.random.default_rng(26)
    n = 37
    x = rng.standard_normal((2, n)).astype(np.float32)
    g = (1.0 + np.arange(n) / 8.0).astype(np.float32)
    b = (np.arange(n) / 16.0 - 1.0).astype(np.float32)
    plain = orc.layernorm(F32, x, wide=True)["y_wide"]
    aff = orc.layernorm(F32, x, g, b, wide=True)["y_wide"]
    assert np.max(np.abs(aff - (plain * g + b))) <= 1e-12


def pin_ln_storage_rounding(orc):
    # y in storage type == RN(y_wide) by an independent conversion
    rng = np.random.default_rng(27)
    for dt in (F16, BF16):
        x = _enc(dt, rng.integers(-255, 256, size=(3, 96)) / 32.0)
        g = _enc(dt, 1.0 + rng.integers(-8, 9, 96) / 16.0)
        r = orc.layernorm(dt, x, g, None, wide=True)
        if dt == F16:
            ref = B.f64_to_bits_numpy_f16(r["y_wide"])
        else:
            # double -> bf16 directly (exact Decimal-free route: via Fraction compare)
            ref = np.array([_bf16_rn_exact(v) for v in r["y_wide"].ravel()],
                           np.uint16).reshape(r["y_wide"].shape)
        assert np.array_equal(r["y"], ref)


def _bf16_rn_exact(v):
    """Nearest bfloat16 by exhaustive neighbour comparison with Fractions."""
    f = np.float32(v)                  # within one binary32 ulp of v
    cand = B.f32_to_bits_torch_bf16(np.array([f], np.float32))[0]
    best, bestd = None, None
    for c in (int(cand) - 1, int(cand), int(cand) + 1):
        c &= 0xFFFF
        cv = B.bf16_bits_to_f64(np.uint16(c))
        if not np.isfinite(cv):
            continue
        dist = abs(Fraction(float(cv)) - Fraction(float(v)))
        if bestd is None or dist < bestd or (dist == bestd and (c & 1) == 0):
            best, bestd = c, dist
    return best


# --------------------------------------------------------------------------
# RMSNorm and residual-add + RMSNorm
# --------------------------------------------------------------------------
def pin_rms_pm1_pattern(orc):
    rng = np.random.default_rng(31)
    n = 256
    x = np.where(rng.random((3, n)) < 0.5, -1.0, 1.0)
    w = 1.0 + rng.integers(-16, 17, n) / 64.0
    eps = np.float32(1e-6)
    for dt in (F32, F16, BF16):
        r = orc.rmsnorm(dt, _enc(dt, x), _enc(dt, w), eps=eps, wide=True)
        expect = x * w / np.sqrt(1.0 + float(eps))
        assert np.max(np.abs(r["y_wide"] - expect)) <= 1e-15
        assert np.allclose(r["rstd"], 1.0 / np.sqrt(1.0 + float(eps)), rtol=1e-15, atol=0)


def pin_rms_constant(orc):
    eps = np.float32(1e-6)
    for c in (0.5, -3.0, 1000.0):
        x = np.full((2, 33), c)
        w = 1.0 + np.arange(33) / 32.0
        r = orc.rmsnorm(F32, _enc(F32, x), _enc(F32, w), eps=eps, wide=True)
        expect = c / np.sqrt(c * c + float(eps)) * w
        assert np.max(np.abs(r["y_wide"] - expect)) <= 1e-14


def pin_rms_scaling_eps0(orc):
    rng = np.random.default_rng(32)
    x = rng.integers(-1000, 1000, size=(3, 77)) / 64.0
    a = orc.rmsnorm(F32, _enc(F32, x), eps=np.float32(0.0), wide=True)["y_wide"]
    b = orc.rmsnorm(F32, _enc(F32, x * 4.0), eps=np.float32(0.0), wide=True)["y_wide"]
    assert np.max(np.abs(a - b)) <= 1e-14
    # exact mean square
    for i in range(3):
        ms = sum(Fraction(float(v)) ** 2 for v in x[i]) / x.shape[1]
        rr = Decimal(1) / (Decimal(ms.numerator) / Decimal(ms.denominator)).sqrt()
        for j in range(0, 77, 7):
            _close(a[i, j], _dec(x[i, j]) * rr, 1e-14, 1e-15)


def pin_add_rms_residual_bits(orc):
    rng = np.random.default_rng(33)
    for dt in (F16, BF16, F32):
        n = 160
        xv = rng.standard_normal((4, n)) * 3
        rv = rng.standard_normal((4, n)) * 2 * 2.0 ** rng.integers(-12, 12, (4, n))
        if dt == F16:
            xb, rb = B.f64_to_bits_numpy_f16(xv), B.f64_to_bits_numpy_f16(rv)
            s = (B.f16_bits_to_f64(xb).astype(np.float32) + B.f16_bits_to_f64(rb).astype(np.float32))
            expect = B.f64_to_bits_numpy_f16(s.astype(np.float64))
        elif dt == BF16:
            xb = B.f32_to_bits_torch_bf16(xv.astype(np.float32))
            rb = B.f32_to_bits_torch_bf16(rv.astype(np.float32))
            s = (B.bf16_bits_to_f64(xb).astype(np.float32) + B.bf16_bits_to_f64(rb).astype(np.float32))
            expect = B.f32_to_bits_torch_bf16(s)
        else:
            xb, rb = xv.astype(np.float32), rv.astype(np.float32)
            expect = xb + rb
        w = _enc(dt, 1.0 + rng.integers(-8, 9, n) / 32.0)
        r = orc.add_rmsnorm(dt, xb, rb, w, eps=np.float32(1e-6), wide=True)
        assert np.array_equal(r["residual_out"], expect)
        # y is RMSNorm of the ROUNDED residual stream (fused RMSNorm page, 3.2)
        v = B.bits_to_f64(dt, r["residual_out"])
        wv = B.bits_to_f64(dt, w)
        for i in range(4):
            ms = sum(Fraction(float(t)) ** 2 for t in v[i]) / n + Fraction(float(np.float32(1e-6)))
            rr = Decimal(1) / (Decimal(ms.numerator) / Decimal(ms.denominator)).sqrt()
            _close(r["rstd"][i], rr, 1e-14)
            for j in range(0, n, 9):
                _close(r["y_wide"][i, j], _dec(v[i, j]) * rr * _dec(wv[j]), 1e-14, 1e-15)


def pin_add_rms_zero_residual_is_rms(orc):
    rng = np.random.default_rng(34)
    for dt in (F16, BF16):
        x = _enc(dt, rng.integers(-255, 256, size=(5, 64)) / 16.0)
        w = _enc(dt, 1.0 + rng.integers(-8, 9, 64) / 16.0)
        zero = np.zeros_like(x)
        a = orc.add_rmsnorm(dt, x, zero, w, eps=np.float32(1e-6))
        b = orc.rmsnorm(dt, x, w, eps=np.float32(1e-6))
        assert np.array_equal(a["residual_out"], x)
        assert np.array_equal(a["y"], b["y"])
        assert np.array_equal(a["rstd"], b["rstd"])


# --------------------------------------------------------------------------
# BatchNorm2d training forward
# --------------------------------------------------------------------------
def pin_bn_arithmetic_channels(orc):
    # x[n, c, k] = a_c + d_c * (n*HW + k): per channel an arithmetic sequence in
    # (n, k) order, with a different (a_c, d_c) per channel, so a wrong NCHW
    # index or a transposed (n, c) shows up in the statistics.
    batch, C, HW = 3, 5, 12
    a = np.array([-2.0, 0.5, 3.0, 10.0, -0.25])
    d = np.array([0.5, 0.25, 1.0, 2.0, 0.125])
    x = np.empty((batch, C, HW))
    for n in range(batch):
        for c in range(C):
            x[n, c] = a[c] + d[c] * (n * HW + np.arange(HW))
    cnt = batch * HW
    m = np.float32(0.1)
    rm0 = np.array([0.5, -1.0, 0.0, 2.0, 1.0])
    rv0 = np.array([1.0, 2.0, 0.5, 1.0, 3.0])
    r = orc.batchnorm_train(F32, _enc(F32, x), running_mean=rm0, running_var=rv0,
                            eps=np.float32(0.0), momentum=m)
    mean = a + d * (cnt - 1) / 2.0
    var = d * d * (cnt * cnt - 1) / 12.0
    for c in range(C):
        _close(r["save_mean"][c], mean[c], 1e-15, 1e-15)
        _close(1.0 / r["save_rstd"][c] ** 2, var[c], 1e-12)
        mm = float(m)
        _close(r["running_mean"][c], (1 - mm) * rm0[c] + mm * mean[c], 1e-14, 1e-15)
        _close(r["running_var"][c], (1 - mm) * rv0[c] + mm * var[c] * cnt / (cnt - 1), 1e-14)


def pin_bn_exact_tiny(orc):
    rng = np.random.default_rng(41)
    batch, C, HW = 2, 3, 4
    x = rng.integers(-40, 41, size=(batch, C, HW)) / 8.0
    g = 1.0 + rng.integers(-8, 9, C) / 8.0
    b = rng.integers(-8, 9, C) / 16.0
    eps = np.float32(1e-5)
    r = orc.batchnorm_train(F32, _enc(F32, x), _enc(F32, g), _enc(F32, b), eps=eps, wide=True)
    for c in range(C):
        vals = x[:, c, :].ravel()
        mean, var, rstd, ys = _exact_ln_row(vals, [g[c]] * vals.size, [b[c]] * vals.size, eps)
        _close(r["save_mean"][c], mean, 1e-15, 1e-15)
        _close(r["save_rstd"][c], rstd, 1e-14)
        got = r["y_wide"][:, c, :].ravel()
        for j in range(vals.size):
            _close(got[j], ys[j], 1e-13, 1e-13)


def pin_bn_single_plane_is_ln(orc):
    rng = np.random.default_rng(42)
    x = (rng.standard_normal((1, 1, 200)) * 2 + 1).astype(np.float32)
    eps = np.float32(1e-5)
    bn = orc.batchnorm_train(F32, x, eps=eps, wide=True)
    ln = orc.layernorm(F32, x.reshape(1, 200), eps=eps, wide=True)
    assert np.max(np.abs(bn["y_wide"].ravel() - ln["y_wide"].ravel())) <= 1e-13


# --------------------------------------------------------------------------
# BatchNorm inference forward (running statistics)
# --------------------------------------------------------------------------
def pin_bn_infer_exact_tiny(orc):
    rng = np.random.default_rng(51)
    batch, C, HW = 2, 3, 5
    x = rng.integers(-40, 41, size=(batch, C, HW)) / 8.0
    g = 1.0 + rng.integers(-8, 9, C) / 8.0
    b = rng.integers(-8, 9, C) / 16.0
    rm = rng.integers(-16, 17, C) / 8.0
    rv = 0.25 + rng.integers(0, 32, C) / 8.0
    eps = np.float32(1e-5)
    for dt in (F32, F16, BF16):
        r = orc.batchnorm_infer(dt, _enc(dt, x), rm.astype(np.float32), rv.astype(np.float32),
                                _enc(dt, g), _enc(dt, b), eps=eps, wide=True)
        for c in range(C):
            den = (_dec(rv[c]) + _dec(eps)).sqrt()
            for n in range(batch):
                for k in range(HW):
                    want = (_dec(x[n, c, k]) - _dec(rm[c])) / den * _dec(g[c]) + _dec(b[c])
                    _close(r["y_wide"][n, c, k], want, 1e-14, 1e-14)


def pin_bn_infer_identity_statistics(orc):
    # running mean 0, running variance 1, eps 0: y = x * gamma + beta exactly
    rng = np.random.default_rng(52)
    batch, C, HW = 3, 4, 6
    x = rng.integers(-64, 65, size=(batch, C, HW)) / 16.0
    g = 1.0 + rng.integers(-8, 9, C) / 8.0
    b = rng.integers(-8, 9, C) / 8.0
    r = orc.batchnorm_infer(F32, _enc(F32, x), np.zeros(C, np.float32), np.ones(C, np.float32),
                            _enc(F32, g), _enc(F32, b), eps=np.float32(0.0), wide=True)
    assert np.array_equal(r["y_wide"], x * g[None, :, None] + b[None, :, None])


def pin_bn_infer_with_batch_statistics_is_train(orc):
    # channels that are arithmetic sequences have a mean and biased variance
    # exact in binary32; feeding them as running statistics reproduces the
    # training forward's normalization
    batch, HW = 2, 8
    cnt = batch * HW
    a = np.array([0.5, -3.0, 10.0])
    d = np.array([0.25, 1.0, 0.5])
    C = a.size
    x = np.empty((batch, C, HW))
    for c in range(C):
        x[:, c, :] = (a[c] + d[c] * np.arange(cnt)).reshape(batch, HW)
    mean = a + d * (cnt - 1) / 2.0
    var = d * d * (cnt * cnt - 1) / 12.0
    assert np.array_equal(mean.astype(np.float32), mean)
    assert np.array_equal(var.astype(np.float32), var)
    eps = np.float32(1e-3)
    inf = orc.batchnorm_infer(F32, _enc(F32, x), mean.astype(np.float32), var.astype(np.float32),
                              eps=eps, wide=True)
    tr = orc.batchnorm_train(F32, _enc(F32, x), eps=eps, wide=True)
    assert np.max(np.abs(inf["y_wide"] - tr["y_wide"])) <= 1e-13


# --------------------------------------------------------------------------
# BatchNorm training backward
# --------------------------------------------------------------------------
def _bn_loss(orc, x, g, b, dy, eps):
    """L = sum(dy * y) with y the training forward of x (double outputs)."""
    r = orc.batchnorm_train(F32, x, g, b, eps=eps, wide=True)
    return float(np.sum(dy * r["y_wide"]))


def pin_bn_bwd_matches_finite_differences(orc):
    # Gradient check (the BatchNorm page's section 6.3 recommends one): the
    # backward of L = sum(dy * y) against central differences of the training
    # forward, which recomputes the batch statistics at every perturbed x.
    # x, gamma and the steps are multiples of 2^-12, so x +- h is exact.
    rng = np.random.default_rng(61)
    batch, C, HW = 2, 2, 3
    x = (rng.integers(-256, 257, size=(batch, C, HW)) / 64.0).astype(np.float32)
    g = (1.0 + rng.integers(-8, 9, C) / 8.0).astype(np.float32)
    b = (rng.integers(-8, 9, C) / 16.0).astype(np.float32)
    dy = rng.standard_normal((batch, C, HW))
    eps = np.float32(1e-2)
    fw = orc.batchnorm_train(F32, x, g, b, eps=eps)
    bw = orc.batchnorm_backward(F32, _enc(F32, np.zeros((batch, C, HW))), x,
                                fw["save_mean"], fw["save_rstd"], g, wide=True)
    h = 2.0 ** -12
    # dy enters the backward as data: use the real dy in double via linearity
    # (the backward is linear in dy: run it once per unit vector of dy)
    grad = np.zeros((batch, C, HW))
    for idx in np.ndindex(batch, C, HW):
        unit = np.zeros((batch, C, HW), np.float32)
        unit[idx] = 1.0
        grad += dy[idx] * orc.batchnorm_backward(F32, unit, x, fw["save_mean"], fw["save_rstd"],
                                                 g, wide=True)["dx_wide"]
    for idx in np.ndindex(batch, C, HW):
        xp = x.copy(); xp[idx] += np.float32(h)
        xm = x.copy(); xm[idx] -= np.float32(h)
        num = (_bn_loss(orc, xp, g, b, dy, eps) - _bn_loss(orc, xm, g, b, dy, eps)) / (2 * h)
        _close(grad[idx], num, 1e-5, 1e-7)
    # dgamma, dbeta: central differences in gamma and beta
    dyf = dy.astype(np.float32)
    full = orc.batchnorm_backward(F32, dyf, x, fw["save_mean"], fw["save_rstd"], g)
    for c in range(C):
        for which, key in ((0, "dgamma"), (1, "dbeta")):
            gp, gm, bp, bm = g.copy(), g.copy(), b.copy(), b.copy()
            if which == 0:
                gp[c] += np.float32(h); gm[c] -= np.float32(h)
            else:
                bp[c] += np.float32(h); bm[c] -= np.float32(h)
            num = (_bn_loss(orc, x, gp, bp, dyf.astype(np.float64), eps)
                   - _bn_loss(orc, x, gm, bm, dyf.astype(np.float64), eps)) / (2 * h)
            _close(full[key][c], num, 1e-6, 1e-7)
    assert np.all(bw["dx_wide"] == 0.0)


def pin_bn_bwd_exact_tiny(orc):
    # sums and dx in 60-digit decimals from the formulas of the BatchNorm
    # page's section 3.1, on binary-fraction data
    rng = np.random.default_rng(62)
    batch, C, HW = 2, 2, 4
    x = rng.integers(-40, 41, size=(batch, C, HW)) / 8.0
    dy = rng.integers(-16, 17, size=(batch, C, HW)) / 8.0
    g = 1.0 + rng.integers(-8, 9, C) / 8.0
    mean = rng.integers(-8, 9, C) / 4.0
    rstd = 0.5 + rng.integers(0, 8, C) / 4.0
    r = orc.batchnorm_backward(F32, _enc(F32, dy), _enc(F32, x), mean, rstd, _enc(F32, g),
                               wide=True)
    cnt = batch * HW
    for c in range(C):
        xh = [(_dec(x[n, c, k]) - _dec(mean[c])) * _dec(rstd[c])
              for n in range(batch) for k in range(HW)]
        dd = [_dec(dy[n, c, k]) for n in range(batch) for k in range(HW)]
        s1 = sum(dd)
        s2 = sum(a * b for a, b in zip(dd, xh))
        _close(r["dbeta"][c], s1, 1e-15, 1e-15)
        _close(r["dgamma"][c], s2, 1e-15, 1e-15)
        j = 0
        for n in range(batch):
            for k in range(HW):
                want = _dec(g[c]) * _dec(rstd[c]) * (dd[j] - s1 / cnt - xh[j] * s2 / cnt)
                _close(r["dx_wide"][n, c, k], want, 1e-14, 1e-14)
                j += 1


def pin_bn_bwd_invariants(orc):
    # with the batch's own statistics: sum over a channel of dx is 0, a
    # constant dy gives dx = 0 and dbeta = k * count, and with eps = 0
    # dx is orthogonal to xhat as well
    rng = np.random.default_rng(63)
    batch, C, HW = 3, 4, 10
    x = (rng.standard_normal((batch, C, HW)) * 2 + 1).astype(np.float32)
    g = (1.0 + 0.1 * rng.standard_normal(C)).astype(np.float32)
    dy = rng.standard_normal((batch, C, HW)).astype(np.float32)
    eps = np.float32(0.0)
    fw = orc.batchnorm_train(F32, x, eps=eps)
    r = orc.batchnorm_backward(F32, dy, x, fw["save_mean"], fw["save_rstd"], g, wide=True)
    xh = (x.astype(np.float64) - fw["save_mean"][None, :, None]) * fw["save_rstd"][None, :, None]
    scale = np.abs(r["dx_wide"]).sum(axis=(0, 2))
    assert np.all(np.abs(r["dx_wide"].sum(axis=(0, 2))) <= 1e-13 * scale)
    assert np.all(np.abs((r["dx_wide"] * xh).sum(axis=(0, 2))) <= 1e-13 * scale * 4)
    k = np.float32(0.75)
    rc = orc.batchnorm_backward(F32, np.full_like(dy, k), x, fw["save_mean"], fw["save_rstd"],
                                g, wide=True)
    assert np.max(np.abs(rc["dx_wide"])) <= 1e-14
    assert np.allclose(rc["dbeta"], float(k) * batch * HW, rtol=1e-15, atol=0)
    assert np.max(np.abs(rc["dgamma"])) <= 1e-12


# --------------------------------------------------------------------------
# Row softmax
# --------------------------------------------------------------------------
def pin_softmax_constant_rows(orc):
    for dt in (F32, F16, BF16):
        for n in (1, 7, 64, 1000):
            for c in (0.0, -3.5, 1000.0):
                r = orc.softmax(dt, _enc(dt, np.full((2, n), c)), wide=True)
                assert np.all(r["y_wide"] == 1.0 / n)
                assert np.all(r["row_max"] == c) and np.all(r["row_sum"] == n)


def pin_softmax_exact_tiny(orc):
    # 60-digit evaluation of exp(x_i - max) / sum_j exp(x_j - max)
    rng = np.random.default_rng(71)
    x = rng.integers(-64, 65, size=(3, 9)) / 8.0
    r = orc.softmax(F32, _enc(F32, x), wide=True)
    for i in range(x.shape[0]):
        m = max(_dec(v) for v in x[i])
        e = [(_dec(v) - m).exp() for v in x[i]]
        d = sum(e)
        _close(r["row_max"][i], m, 0.0, 0.0)
        _close(r["row_sum"][i], d, 1e-15)
        for j in range(x.shape[1]):
            _close(r["y_wide"][i, j], e[j] / d, 1e-14, 1e-300)


def pin_softmax_two_values_logistic(orc):
    # a row (a, b) gives y_0 = 1 / (1 + exp(b - a))
    for a, b in ((0.0, 1.0), (2.5, -1.5), (30.0, 30.5), (-7.0, 9.0)):
        r = orc.softmax(F32, _enc(F32, np.array([[a, b]])), wide=True)
        want = Decimal(1) / (Decimal(1) + (_dec(b) - _dec(a)).exp())
        _close(r["y_wide"][0, 0], want, 1e-15)
        _close(r["y_wide"][0, 1], Decimal(1) - want, 1e-14)


def pin_softmax_shift_and_overflow(orc):
    # softmax(x + c) = softmax(x); large inputs stay finite (the max is
    # subtracted before exp); outputs sum to 1
    rng = np.random.default_rng(72)
    base = rng.integers(-512, 513, size=(4, 200)) / 32.0
    ref = orc.softmax(F32, _enc(F32, base), wide=True)["y_wide"]
    for c in (1000.0, -600.0, 5000.0):
        got = orc.softmax(F32, _enc(F32, base + c), wide=True)["y_wide"]
        assert np.all(np.isfinite(got))
        assert np.max(np.abs(got - ref)) <= 1e-15
    assert np.max(np.abs(ref.sum(axis=1) - 1.0)) <= 1e-14


def pin_softmax_online_recurrence_matches(orc):
    # The single-pass update of the LLM-ops page (section 1, "online softmax"):
    # m_new = max(m_old, x_k), d_new = d_old * exp(m_old - m_new) + exp(x_k - m_new),
    # run in Python doubles, reaches the oracle's max and denominator; and the
    # page's pairwise merge of two (max, sum) halves reaches the same pair.
    rng = np.random.default_rng(73)
    x = (rng.standard_normal((5, 333)) * 4).astype(np.float32)
    r = orc.softmax(F32, x)
    for i in range(x.shape[0]):
        m, d = float("-inf"), 0.0
        for v in x[i].astype(np.float64):
            mn = max(m, v)
            d = d * np.exp(m - mn) + np.exp(v - mn)
            m = mn
        _close(r["row_max"][i], m, 0.0, 0.0)
        _close(r["row_sum"][i], d, 1e-13)
        h = x.shape[1] // 2
        lo, hi = x[i, :h].astype(np.float64), x[i, h:].astype(np.float64)
        ma, mb = lo.max(), hi.max()
        da, db = np.exp(lo - ma).sum(), np.exp(hi - mb).sum()
        mm = max(ma, mb)
        _close(r["row_sum"][i], da * np.exp(ma - mm) + db * np.exp(mb - mm), 1e-13)


def pin_softmax_ratios_and_rounding(orc):
    # y_i / y_j = exp(x_i - x_j); 16-bit outputs are the nearest value of y
    rng = np.random.default_rng(74)
    x = rng.integers(-96, 97, size=(3, 50)) / 16.0
    r = orc.softmax(F32, _enc(F32, x), wide=True)
    y = r["y_wide"]
    for i in range(3):
        j, k = int(np.argmax(x[i])), int(np.argmin(x[i]))
        _close(y[i, k] / y[i, j], np.exp(x[i, k] - x[i, j]), 1e-13)
    for dt in (F16, BF16):
        rr = orc.softmax(dt, _enc(dt, x), wide=True)
        if dt == F16:
            ref = B.f64_to_bits_numpy_f16(rr["y_wide"])
        else:
            ref = np.array([_bf16_rn_exact(v) for v in rr["y_wide"].ravel()],
                           np.uint16).reshape(rr["y_wide"].shape)
        assert np.array_equal(rr["y"], ref)


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
