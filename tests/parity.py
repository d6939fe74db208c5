"""Comparison helpers for GPU-vs-oracle parity (test infrastructure).

Rules (thresholds also printed by bench.py):
  * page tables, BF16 sink / ring bytes: exact;
  * fp16 s and z: exact, except one fp16 ulp where the oracle's fp32 value
    (min, or (max - min) / 3) lies within 1e-5 relative of an fp16 rounding
    midpoint -- then the group's codes are re-derived from the oracle's fp32
    rotated values with the GPU's s and z;
  * 2-bit codes: exact, except one step where the oracle's t = (x - z) / s
    lies within 1e-5 * max(1, |t|) of a rounding boundary k + 1/2;
  * attention output: max-abs <= 1e-2 and ||diff||_F / ||ref||_F <= 5e-3.
"""
from __future__ import annotations

import numpy as np

from oracle import layout, quant

OUT_MAX_ABS = 1e-2
OUT_REL_FRO = 5e-3
BAND = 1e-5


def near_fp16_midpoint(v32: np.ndarray) -> np.ndarray:
    """True where an fp32 value is within BAND (relative) of an fp16 rounding midpoint."""
    v = np.asarray(v32, dtype=np.float64)
    h = v.astype(np.float16).astype(np.float64)
    up = np.nextafter(h.astype(np.float16), np.float16(np.inf)).astype(np.float64)
    dn = np.nextafter(h.astype(np.float16), np.float16(-np.inf)).astype(np.float64)
    mid = np.where(v >= h, (h + up) / 2, (h + dn) / 2)
    return np.abs(v - mid) <= BAND * np.maximum(np.abs(v), 1e-30)


def _t_near_boundary(t: np.ndarray) -> np.ndarray:
    # t is nan / inf in a constant group (s = 0), whose codes are all 0 on both sides
    with np.errstate(invalid="ignore"):
        frac = t - np.floor(t)
    return (np.abs(frac - 0.5) <= BAND * np.maximum(1.0, np.abs(t))) & (t > 0) & (t < 3)


def compare_groups(gpu_packed, gpu_meta, x32, tau, group=128):
    """Compare GPU code bytes [n][32] and meta [n][4 * groups] of one head / K-or-V
    with the oracle.

    x32: oracle fp32 rotated values [n][128].  With group = 64 every token-head is
    two groups, compared as rows of their own.  Returns a dict of counts; raises
    AssertionError on any out-of-band difference.
    """
    x32 = np.asarray(x32, np.float32).reshape(-1, group)
    tau = np.float32(tau)
    codes_o, s_o, z_o = quant.quantize_groups(x32, tau, group)
    s_g, z_g = layout.meta_to_sz(np.asarray(gpu_meta, np.uint8).reshape(-1, 4))
    codes_g = layout.unpack_codes(np.asarray(gpu_packed, np.uint8)).reshape(-1, group)
    xc = (np.minimum(np.maximum(x32, -tau), tau) + np.float32(0)).astype(np.float32)
    mn = xc.min(1)
    mx = xc.max(1)
    r = ((mx - mn).astype(np.float32) / np.float32(3)).astype(np.float32)
    sb_o, sb_g = s_o.view(np.uint16).astype(np.int64), s_g.view(np.uint16).astype(np.int64)
    zb_o, zb_g = z_o.view(np.uint16).astype(np.int64), z_g.view(np.uint16).astype(np.int64)
    s_diff = sb_o != sb_g
    z_diff = zb_o != zb_g
    s_ok = ~s_diff | ((np.abs(sb_o - sb_g) == 1) & near_fp16_midpoint(r))
    z_ok = ~z_diff | ((np.abs(zb_o - zb_g) == 1) & near_fp16_midpoint(mn))
    bad_meta = np.nonzero(~(s_ok & z_ok))[0]
    assert bad_meta.size == 0, f"meta out of band in groups {bad_meta[:8]}: s {sb_o[bad_meta[:4]]} vs " \
                               f"{sb_g[bad_meta[:4]]}, z {zb_o[bad_meta[:4]]} vs {zb_g[bad_meta[:4]]}"
    # reference codes: oracle's own, or re-derived with the GPU's s / z where those were exempted
    meta_exempt = s_diff | z_diff
    ref_codes = codes_o.copy()
    t = quant.t_values(x32, tau, s_o, z_o)
    if meta_exempt.any():
        idx = np.nonzero(meta_exempt)[0]
        c2, _, _ = _codes_with(xc[idx], s_g[idx], z_g[idx])
        ref_codes[idx] = c2
        t[idx] = quant.t_values(x32[idx], tau, s_g[idx], z_g[idx])
    diff = ref_codes.astype(np.int64) - codes_g.astype(np.int64)
    mism = diff != 0
    exempt = mism & (np.abs(diff) == 1) & _t_near_boundary(t)
    bad = mism & ~exempt
    assert not bad.any(), f"{int(bad.sum())} codes out of band, first at {np.argwhere(bad)[:4].tolist()}"
    return {"groups": int(x32.shape[0]), "codes": int(codes_o.size), "code_exempt": int(exempt.sum()),
            "meta_exempt": int(meta_exempt.sum())}


def _codes_with(xc, s, z):
    zf = z.astype(np.float32)[:, None]
    sf = s.astype(np.float32)[:, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        t = ((xc - zf).astype(np.float32) / sf).astype(np.float32)
    c = np.clip(np.rint(t), 0, 3)
    c = np.where(sf == 0, 0, c)
    return c.astype(np.uint8), s, z


def check_output(got: np.ndarray, ref: np.ndarray):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    max_abs = float(np.abs(got - ref).max())
    rel = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))
    assert max_abs <= OUT_MAX_ABS and rel <= OUT_REL_FRO, f"max_abs {max_abs:.3e} rel_fro {rel:.3e}"
    return {"max_abs": max_abs, "rel_fro": rel}


def slot_bytes(records, rows: int, group: int = 128) -> np.ndarray:
    """What token slots 0..rows-1 of page-head records hold, uint8 [heads][...]:
    their K and V codes and K / V meta.  Slots past ``rows`` (never written,
    arbitrary) are left out, so two caches compare equal exactly when their
    written tokens do."""
    recs = np.asarray(records, dtype=np.uint8)
    out = []
    for rec in recs.reshape(-1, recs.shape[-1]):
        f = [layout.record_slot_fields(rec, r, group) for r in range(rows)]
        out.append(np.concatenate([np.concatenate(x) for x in zip(*f)]) if rows else np.zeros(0, np.uint8))
    return np.stack(out)


def bf16_to_f64(t) -> np.ndarray:
    """torch bf16 tensor (any device) -> float64 numpy."""
    import torch
    return t.detach().to(torch.float32).cpu().numpy().astype(np.float64)
