"""Rotation ablation on the GPU path: naive INT2, Hadamard only, and OSCAR.

"Together AI Open-Sources OSCAR" (MarkTechPost), section "What OSCAR Does
Differently": quantising keys in their own basis (naive INT2) lets a few outlier
channels and the query-blind grid dominate the error; a Hadamard rotation
spreads the outliers; OSCAR's R_K = U_Q H P_br also aligns the grid with the
query covariance (and R_V = U_S H P_br with the score-weighted values), which
is what its attention-error tables measure.

For one seeded synthetic layer, each variant fits its clip thresholds on the
same calibration set, prefills a cache through the C ABI and decodes the same queries.  Against
exact attention over the BF16 tokens (float64 on the host) it reports:
  * logit_rel: |S - S^|_F / |S|_F of the scaled scores q k^T / sqrt(d) over the
    INT2 history, with K^ dequantised from the cache's own bytes
    (x^ = z + s c in the rotated basis, times R_K^T);
  * kl: mean KL(softmax(S) || softmax(S^)) over query heads and queries, all
    tokens (the BF16 segments are exact on both sides);
  * out_rel, out_max_abs: the decode call's outputs.
The same page says the permuted bit-reversal P_br spreads every importance
level over the quantisation groups, which only matters with more than one group
per token-head: the "_nobr" variants drop it (R = H, R = U H) to measure that at
G_K = 64.
Two laws (synth.py): "outliers", the workloads' law (K / V with x20 outlier
channels, queries from N(0, Sigma) with a full-rank Wishart Sigma), and
"subspace", where the queries of a GQA group have four dominant eigen-directions
that the keys share (x5 outlier channels).  On the first a Hadamard rotation
alone already gives every channel the same query importance (the outliers are
axis-aligned), so the query eigenbasis has nothing to add; the second is the
structure the query-covariance alignment is for.
Usage: ``python -m bit_rotated_kv_decode_gb300.ablation``.
"""
from __future__ import annotations

import json

import numpy as np

from . import calibrate, synth

VARIANTS = ("naive", "hadamard", "oscar")
BR_VARIANTS = ("hadamard_nobr", "hadamard", "oscar_nobr", "oscar")


def rotations(variant: str, q_cal, k_cal, v_cal, hkv: int, clip: float):
    """fp32 R_K, R_V [H_kv][d][d] and tau_K, tau_V [H_kv] of one variant."""
    d = synth.HEAD_DIM
    if variant in ("oscar", "oscar_nobr"):
        return calibrate.calibrate_layer(q_cal, k_cal, v_cal, clip, clip, bit_reversal=variant == "oscar")
    if variant in ("hadamard", "hadamard_nobr"):
        r = calibrate.composed_rotation(np.eye(d), bit_reversal=variant == "hadamard").astype(np.float32)
    elif variant == "naive":
        r = np.eye(d, dtype=np.float32)
    else:
        raise ValueError(variant)
    rk = np.broadcast_to(r, (hkv, d, d)).copy()
    rv = rk.copy()
    tk = np.array([np.quantile(np.abs(k_cal[:, h] @ r.astype(np.float64)), clip, method="linear")
                   for h in range(hkv)], dtype=np.float32)
    tv = np.array([np.quantile(np.abs(v_cal[:, h] @ r.astype(np.float64)), clip, method="linear")
                   for h in range(hkv)], dtype=np.float32)
    return rk, rv, tk, tv


def exact_attention(q, k, v, hkv: int):
    """float64 softmax(q k^T / sqrt(d)) v for q [Hq][d], k, v [T][H_kv][d]."""
    hq, d = q.shape
    g = hq // hkv
    out = np.empty((hq, d))
    for h in range(hq):
        kh, vh = k[:, h // g], v[:, h // g]
        s = kh @ q[h] / np.sqrt(d)
        p = np.exp(s - s.max())
        out[h] = (p @ vh) / p.sum()
    return out


def dequantised_keys(pool, hist_pages, nhist: int, rk, hkv: int, group: int = 128):
    """K^ [nhist][H_kv][d] (float64) from INT2 records [pages][H_kv][4608 or 5120] (uint8):
    per group of ``group`` channels, x = z + s c from that group's {s, z}."""
    d = synth.HEAD_DIM
    ng = d // group
    out = np.empty((nhist, hkv, d))
    shifts = np.array([0, 2, 4, 6], dtype=np.uint8)
    for h in range(nhist):
        rec = pool[hist_pages[h // 64]]                 # [H_kv][record]
        row = h % 64
        codes = rec[:, 32 * row: 32 * row + 32]         # K codes: channel 4 j + i in bits 2 i of byte j
        c = ((codes[:, :, None] >> shifts) & 3).reshape(hkv, ng, group).astype(np.float64)
        meta = rec[:, 4096 + 4 * ng * row: 4096 + 4 * ng * (row + 1)].copy().view(np.float16).astype(np.float64)
        meta = meta.reshape(hkv, ng, 2)                 # per group {s, z}
        x = (meta[:, :, 1:2] + meta[:, :, 0:1] * c).reshape(hkv, d)
        out[h] = np.einsum("hc,hic->hi", x, rk.astype(np.float64))   # x R^T: row i of R times x
    return out


def run(cfg_id: int = 0, hq: int = 32, hkv: int = 8, tokens: int = 8192, queries: int = 8, clip: float = 0.9,
        layer: int = 0, group: int = 128, variants=VARIANTS, law: str = "outliers") -> dict:
    """law: "outliers" (the workloads' law: x20 outlier channels, full-rank query
    covariance) or "subspace" (queries and keys sharing a 4-dimensional dominant
    subspace, x5 outlier channels)."""
    import torch

    from . import binding
    binding.load()
    d = synth.HEAD_DIM
    if law == "outliers":
        q_cal, k_cal, v_cal = synth.calibration_set(cfg_id, layer, hq, hkv, 512)
        k = synth.kv_tokens(cfg_id, layer, hkv, "k", range(tokens), device="cuda")
        v = synth.kv_tokens(cfg_id, layer, hkv, "v", range(tokens), device="cuda")
        qs = [synth.queries(cfg_id, layer, hq, 1, step, device="cuda") for step in range(queries)]
    elif law == "subspace":
        q_cal, k_cal, v_cal = synth.subspace_calibration_set(cfg_id, layer, hq, hkv, 512)
        k = synth.subspace_kv(cfg_id, layer, hkv, "k", tokens, device="cuda")
        v = synth.subspace_kv(cfg_id, layer, hkv, "v", tokens, device="cuda")
        qs = [synth.subspace_queries(cfg_id, layer, hq, hkv, 1, step, device="cuda") for step in range(queries)]
    else:
        raise ValueError(law)
    kf = k.float().cpu().numpy().astype(np.float64)
    vf = v.float().cpu().numpy().astype(np.float64)
    refs = [exact_attention(q[0].float().cpu().numpy().astype(np.float64), kf, vf, hkv) for q in qs]
    pages = (tokens - 320) // 64 + 2
    results = {}
    for variant in variants:
        rk, rv, tk, tv = rotations(variant, q_cal, k_cal, v_cal, hkv, clip)
        cfg = binding.make_config(1, hq, hkv, 1, pages, pages + 2, 0, 0.0, 0, group_size=group)
        cache = binding.OscarCache(cfg, torch.from_numpy(rk).cuda(), torch.from_numpy(rv).cuda(), tk, tv)
        r = cache.open()
        cache.prefill(r, 0, k, v)
        ws = binding.new_workspace(cache.workspace_bytes([r]))
        nhist = tokens - 320
        kq = dequantised_keys(cache.int2_pool(0).cpu().numpy(), cache.pages(r)[0], nhist, rk, hkv, group)
        khat = kf.copy()
        khat[64:64 + nhist] = kq
        g = hq // hkv
        lnum = lden = kl = 0.0
        for q in qs:
            qf = q[0].float().cpu().numpy().astype(np.float64)
            for h in range(hq):
                s_ex = kf[:, h // g] @ qf[h] / np.sqrt(d)
                s_q = khat[:, h // g] @ qf[h] / np.sqrt(d)
                lnum += float(((s_q - s_ex)[64:64 + nhist] ** 2).sum())
                lden += float((s_ex[64:64 + nhist] ** 2).sum())
                a = s_ex - s_ex.max()
                b = s_q - s_q.max()
                la = a - np.log(np.exp(a).sum())
                lb = b - np.log(np.exp(b).sum())
                kl += float((np.exp(la) * (la - lb)).sum())
        num = den = 0.0
        max_abs = 0.0
        for q, ref in zip(qs, refs):
            out = torch.empty((1, hq, d), dtype=torch.float32, device="cuda")
            cache.decode(0, [r], q, out, ws)
            got = out[0].cpu().numpy().astype(np.float64)
            num += float(((got - ref) ** 2).sum())
            den += float((ref ** 2).sum())
            max_abs = max(max_abs, float(np.abs(got - ref).max()))
        cache.check()
        cache.close(r)
        results[variant] = {"logit_rel": (lnum / lden) ** 0.5, "kl": kl / (len(qs) * hq),
                            "out_rel": (num / den) ** 0.5, "out_max_abs": max_abs}
    return {"config": {"cfg_id": cfg_id, "q_heads": hq, "kv_heads": hkv, "tokens": tokens, "queries": queries,
                       "clip": clip, "layer": layer, "group": group, "law": law}, "results": results}


if __name__ == "__main__":
    for clip in (1.0, 0.9):
        print(json.dumps(run(clip=clip)))
    # the bit-reversal's share, with one group and with two groups per token-head
    for group in (128, 64):
        print(json.dumps(run(clip=0.9, group=group, variants=BR_VARIANTS)))
    # queries with a few dominant directions that the keys share
    for group in (128, 64):
        print(json.dumps(run(clip=0.9, group=group, variants=BR_VARIANTS + ("naive",), law="subspace")))
