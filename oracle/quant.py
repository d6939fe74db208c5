"""Rotate, clip, quantise to INT2 (oracle; test infrastructure).

[MTP] section "The Serving System: Mixed-Precision Cache Layout": on the write
path each token is rotated, clipped to a calibration-derived threshold, then
quantised with per-token asymmetric INT2.  [MS] section "OSCAR的设计": the read
side dequantises with a scale and a zero point; [MS] section "快速实践": group
size 128 (``--kv-cache-quant-group-size 128``), i.e. one group per token-head;
[MTP] section "What OSCAR Does Differently" names G_K = 64 channels per group
as the default, i.e. two groups per token-head, each with its own s and z.

Readings (the pages give no formula):
  * x = k . R evaluated exactly, then rounded once to fp32 -- fp32 is the
    precision the kernels take every quantisation decision in, so the oracle
    takes them in fp32 too;
  * clip: x <- min(max(x, -tau), tau) with the stored fp32 tau, then + 0 so a
    signed zero becomes +0 (IEEE: -0 + +0 = +0) and min/max are unambiguous;
  * z = fp16_rn(min x), s = fp16_rn(fl32(fl32(max x - min x) / 3));
  * code = clamp(rint_half_even(fl32(fl32(x - z) / s)), 0, 3), code = 0 when
    s == 0;
  * dequantised value x_hat = z + s * code (exact real arithmetic);
  * with G_K = 64, every step above is taken per group of 64 consecutive
    rotated channels (0..63 and 64..127), independently.
Every fp32 / fp16 operation above is IEEE round-to-nearest-even.  Pinned by
closed-form groups, round-half-even ties, brute-force nearest-level search and
the reconstruction error bound (tests/test_oracle_quant.py).
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np

LEVELS = 4
MAX_CODE = LEVELS - 1


def _round_fraction_to_fp32(v: Fraction) -> np.float32:
    """Correctly rounded (nearest, ties to even) fp32 of an exact rational."""
    c = np.float32(float(v))
    best = None
    for cand in (np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))):
        err = abs(Fraction(float(cand)) - v)
        even = (int(np.array(cand, dtype=np.float32).view(np.uint32)) & 1) == 0
        key = (err, not even)
        if best is None or key < best[0]:
            best = (key, cand)
    return np.float32(best[1])


def rotate_to_fp32(x: np.ndarray, r: np.ndarray) -> np.ndarray:
    """fp32_rn(x . R) for every row of x, with the exact dot product.

    x: [..., d] float64 holding bf16 values; r: [d][d] float64 holding fp32
    values.  Each product is exact in float64 (8 + 24 significant bits); the
    float64 matmul is exact to within a bound, and the rows whose float64
    result lies too close to an fp32 rounding midpoint are recomputed with
    exact rational arithmetic.
    """
    x = np.asarray(x, dtype=np.float64)
    d = r.shape[0]
    y = x @ r
    bound = (2.0 * d * 2.0 ** -53) * (np.abs(x) @ np.abs(r)) + 1e-300
    y32 = y.astype(np.float32)
    up = np.nextafter(y32, np.float32(np.inf)).astype(np.float64)
    dn = np.nextafter(y32, np.float32(-np.inf)).astype(np.float64)
    y32d = y32.astype(np.float64)
    mid_hi = (y32d + up) / 2.0
    mid_lo = (y32d + dn) / 2.0
    unsafe = ~((y - bound > mid_lo) & (y + bound < mid_hi))
    if np.any(unsafe):
        xf = x.reshape(-1, d)
        yf = y32.reshape(-1, d)
        uf = unsafe.reshape(-1, d)
        rows, cols = np.nonzero(uf)
        for i, j in zip(rows, cols):
            acc = Fraction(0)
            for t in range(d):
                if xf[i, t] != 0.0 and r[t, j] != 0.0:
                    acc += Fraction(float(xf[i, t])) * Fraction(float(r[t, j]))
            yf[i, j] = _round_fraction_to_fp32(acc)
        y32 = yf.reshape(y32.shape)
    return y32


def _split(a: np.ndarray, group: int) -> np.ndarray:
    """[..., d] -> [..., d // group, group] (consecutive channels per group)."""
    d = a.shape[-1]
    if group <= 0 or d % group:
        raise ValueError("group size must divide the channel count")
    return a.reshape(a.shape[:-1] + (d // group, group))


def _per_group(meta: np.ndarray, codes_shape) -> np.ndarray:
    """s or z as [..., groups, 1]: one group when meta has one axis fewer than the codes."""
    meta = np.asarray(meta)
    if meta.ndim == len(codes_shape) - 1:
        meta = meta[..., None]
    return meta[..., None]


def quantize_groups(x32: np.ndarray, tau: np.float32, group: int = 128):
    """Clip and quantise each group of ``group`` consecutive channels of fp32 values.

    Returns (codes uint8 [..., d], s float16, z float16); s and z are [...] when
    the group is the whole row (d == group), else [..., d // group].
    """
    x32 = np.asarray(x32, dtype=np.float32)
    tau = np.float32(tau)
    xc = (np.minimum(np.maximum(x32, -tau), tau) + np.float32(0.0)).astype(np.float32)
    xg = _split(xc, group)
    mn = xg.min(axis=-1)
    mx = xg.max(axis=-1)
    z = mn.astype(np.float16)
    rng = (mx - mn).astype(np.float32)
    s = (rng / np.float32(3.0)).astype(np.float32).astype(np.float16)
    zf = z.astype(np.float32)[..., None]
    sf = s.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        t = ((xg - zf).astype(np.float32) / sf).astype(np.float32)
    code = np.clip(np.rint(t), 0, MAX_CODE)
    code = np.where(sf == 0, 0, code).reshape(xc.shape)
    if xg.shape[-2] == 1:
        s, z = s[..., 0], z[..., 0]
    return code.astype(np.uint8), s, z


def t_values(x32: np.ndarray, tau: np.float32, s: np.ndarray, z: np.ndarray) -> np.ndarray:
    """The fp32 t = (clip(x) - z) / s each code was rounded from (for exemption bands).

    s, z as returned by quantize_groups (one group per row, or [..., groups])."""
    tau = np.float32(tau)
    x32 = np.asarray(x32, np.float32)
    xc = (np.minimum(np.maximum(x32, -tau), tau) + np.float32(0.0)).astype(np.float32)
    zf = _per_group(z, x32.shape).astype(np.float32)
    sf = _per_group(s, x32.shape).astype(np.float32)
    xg = _split(xc, x32.shape[-1] // zf.shape[-2])
    with np.errstate(divide="ignore", invalid="ignore"):
        return ((xg - zf).astype(np.float32) / sf).astype(np.float32).reshape(x32.shape)


def dequantize(codes: np.ndarray, s: np.ndarray, z: np.ndarray) -> np.ndarray:
    """x_hat = z + s * code in float64, per group (s, z as from quantize_groups)."""
    codes = np.asarray(codes)
    zf = _per_group(z, codes.shape).astype(np.float64)
    sf = _per_group(s, codes.shape).astype(np.float64)
    cg = _split(codes.astype(np.float64), codes.shape[-1] // zf.shape[-2])
    return (zf + sf * cg).reshape(codes.shape)


def quantize_tokens(x: np.ndarray, r: np.ndarray, tau: np.float32, group: int = 128):
    """Rotate (exact, rounded to fp32), clip and quantise token rows of one head."""
    x32 = rotate_to_fp32(x, r)
    codes, s, z = quantize_groups(x32, tau, group)
    return codes, s, z, x32
