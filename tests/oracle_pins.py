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


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
