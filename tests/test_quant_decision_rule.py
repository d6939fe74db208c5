"""The division-free code decision of the kernels' quantiser, checked on the host.

The kernels decide a code for an interval [lo, hi] of rotated values from
q' = fl32(fl32(v - z) * r), r an approximate reciprocal of s with at most one
ulp of error, and a margin M = (|q'| + 1) 2^-19: when floor(q'_lo - M + 1/2) and
floor(q'_hi + M + 1/2), clamped to [0, 3], agree, that is the code of every value
in the interval; otherwise the IEEE quotient decides.  The reading fixes the
code as clamp(rint(fl32(fl32(v - z) / s)), 0, 3).  Here the rule runs in numpy
float32 with r taken at both ends of its error range, on random and on
adversarial values (quotients near k + 1/2, tiny and huge scales), and every
decided code must equal the IEEE one.
"""
import numpy as np

F = np.float32


def ieee_code(v, z, s):
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        t = ((v - z).astype(F) / s).astype(F)
        c = np.clip(np.rint(t), 0, 3)
    return np.where(s == 0, 0, c)


def fast_code(lo, hi, z, s, r):
    with np.errstate(over="ignore", invalid="ignore"):
        qa = ((lo - z).astype(F) * r).astype(F)
        qb = ((hi - z).astype(F) * r).astype(F)
        ma = ((np.abs(qa) + F(1)).astype(F) * F(2.0 ** -19)).astype(F)
        mb = ((np.abs(qb) + F(1)).astype(F) * F(2.0 ** -19)).astype(F)
        ca = np.clip(np.floor(((qa - ma).astype(F) + F(0.5)).astype(F)), 0, 3)
        cb = np.clip(np.floor(((qb + mb).astype(F) + F(0.5)).astype(F)), 0, 3)
    return ca, cb


def reciprocals(s):
    """1/s rounded to fp32, and one ulp either side (the approximation's range)."""
    r = (F(1) / s).astype(F)
    return [np.nextafter(r, F(0)), r, np.nextafter(r, F(np.inf))]


def check(lo, hi, z, s):
    decided_total = 0
    for r in reciprocals(s):
        ca, cb = fast_code(lo, hi, z, s, r)
        decided = ca == cb
        want_lo, want_hi = ieee_code(lo, z, s), ieee_code(hi, z, s)
        # decided: every value of [lo, hi] has that code, so both ends do
        assert np.all(want_lo[decided] == ca[decided])
        assert np.all(want_hi[decided] == ca[decided])
        decided_total += int(decided.sum())
    return decided_total


def test_random_intervals():
    rng = np.random.default_rng(0)
    n = 200_000
    s = rng.uniform(1e-3, 4.0, n).astype(np.float16).astype(F)
    z = rng.normal(0, 3, n).astype(np.float16).astype(F)
    t = rng.uniform(-0.3, 3.3, n)
    v = (z.astype(np.float64) + t * s.astype(np.float64)).astype(F)
    e = (np.abs(v) * rng.uniform(0, 2e-6, n)).astype(F)
    lo, hi = (v - e).astype(F), (v + e).astype(F)
    assert check(lo, hi, z, s) > 0.95 * 3 * n          # nearly every interval is decided fast


def test_quotients_at_rounding_boundaries():
    # v chosen so that (v - z) / s sits on or within a few ulps of k + 1/2
    rng = np.random.default_rng(1)
    n = 50_000
    s = rng.uniform(1e-2, 2.0, n).astype(np.float16).astype(F)
    z = rng.normal(0, 1, n).astype(np.float16).astype(F)
    k = rng.integers(0, 3, n)
    v = (z.astype(np.float64) + (k + 0.5) * s.astype(np.float64)).astype(F)
    for steps in (-3, -1, 0, 1, 3):
        w = v.copy()
        for _ in range(abs(steps)):
            w = np.nextafter(w, F(np.inf) if steps > 0 else F(-np.inf))
        check(w, w, z, s)
        check(w, np.nextafter(w, F(np.inf)), z, s)


def test_extreme_scales_and_zero_scale():
    rng = np.random.default_rng(2)
    n = 20_000
    for lo_s, hi_s in ((2.0 ** -24, 2.0 ** -14), (100.0, 6e4)):
        s = rng.uniform(lo_s, hi_s, n).astype(np.float16).astype(F)
        s = np.where(s == 0, F(2.0 ** -24), s)
        z = rng.normal(0, 1, n).astype(np.float16).astype(F)
        v = (z + rng.uniform(-1, 4, n).astype(F) * s).astype(F)
        check(v, v, z, s)
    # s = 0: the kernels take r = 0, so q' = 0 and the code is 0, as defined
    z = np.zeros(10, F)
    s = np.zeros(10, F)
    v = np.linspace(-1, 1, 10).astype(F)
    ca, cb = fast_code(v, v, z, s, np.zeros(10, F))
    assert np.all(ca == 0) and np.all(cb == 0) and np.all(ieee_code(v, z, s) == 0)


def test_device_rule_is_the_rule_checked_here():
    """The kernels' decision (quant_device.cuh) uses the constants and forms of
    fast_code above: an rcp.approx reciprocal, the margin (|q'| + 1) 2^-19, and
    floor(q' -/+ M + 1/2) clamped to [0, 3] at the two ends of the interval."""
    import os
    import re
    src = open(os.path.join(os.path.dirname(__file__), "..", "bit_rotated_kv_decode_gb300", "csrc",
                            "quant_device.cuh")).read()
    assert "rcp.approx.f32" in src
    assert re.search(r"__fmul_rn\(fabsf\(qa\) \+ 1\.0f, 0x1p-19f\)", src)
    assert re.search(r"__fmul_rn\(fabsf\(qb\) \+ 1\.0f, 0x1p-19f\)", src)
    assert re.search(r"fminf\(fmaxf\(floorf\(qa - ma \+ 0\.5f\), 0\.0f\), 3\.0f\)", src)
    assert re.search(r"fminf\(fmaxf\(floorf\(qb \+ mb \+ 0\.5f\), 0\.0f\), 3\.0f\)", src)
    # and this file's restatement uses the same margin
    assert F(2.0 ** -19) == F(float.fromhex("0x1p-19"))

