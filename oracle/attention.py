"""Three-segment decode attention (oracle; test infrastructure).

[MTP] section "The Serving System: Mixed-Precision Cache Layout" and [MS]
section "OSCAR的设计": the cache of one request is a BF16 sink (first 64
tokens), INT2 history, and a BF16 window of recent tokens; decode attends over
all of them (the pages merge a BF16 partial and an INT2 partial with an online
softmax; the result is the softmax over the union, which is what is computed
here directly).

Definition used (plain softmax attention over the reconstructed tokens):
  * BF16 tokens: k~ = k, v~ = v;
  * INT2 tokens: k~ = (z + s c) R_K^T, v~ = (z + s c) R_V^T, with (c, s, z)
    from ``quant.quantize_tokens`` of the raw k, v;
  * logits l_j = scale * q . k~_j (scale 1/sqrt(128) unless given), p =
    softmax(l), out = sum_j p_j v~_j;
  * query head h reads kv head h // G (GQA, G = H_q / H_kv).
Segments: sink = [0, min(T, 64)), history = [64, hist_end), recent =
[hist_end, T) (empty when T <= 64).  With appends only, hist_end =
max(64, T - 256), so the recent window is the last min(256, T - 64) tokens.
Pinned by: equality with plain attention when T <= 320 and when the quantiser
is replaced by the identity; a naive per-token loop; the logit-error identity.
"""
from __future__ import annotations

import numpy as np

from . import quant

SINK = 64


def segments(total: int, hist_end: int):
    sink = range(0, min(total, SINK))
    hist = range(SINK, hist_end) if total > SINK else range(0)
    recent = range(hist_end, total) if total > SINK else range(0)
    return sink, hist, recent


def reconstruct_head(k: np.ndarray, v: np.ndarray, hist_end: int, rk: np.ndarray, rv: np.ndarray,
                     tau_k: float, tau_v: float, identity_quantizer: bool = False, group: int = 128):
    """Keys / values [T][d] float64 as decode sees them, for one kv head."""
    total = k.shape[0]
    kt = np.array(k, dtype=np.float64, copy=True)
    vt = np.array(v, dtype=np.float64, copy=True)
    _, hist, _ = segments(total, hist_end)
    if len(hist):
        idx = np.arange(hist.start, hist.stop)
        if identity_quantizer:
            kt[idx] = (k[idx] @ rk) @ rk.T
            vt[idx] = (v[idx] @ rv) @ rv.T
        else:
            ck, sk, zk, _ = quant.quantize_tokens(k[idx], rk, np.float32(tau_k), group)
            cv, sv, zv, _ = quant.quantize_tokens(v[idx], rv, np.float32(tau_v), group)
            kt[idx] = quant.dequantize(ck, sk, zk) @ rk.T
            vt[idx] = quant.dequantize(cv, sv, zv) @ rv.T
    return kt, vt


def softmax_attention(q: np.ndarray, keys: np.ndarray, values: np.ndarray, scale: float) -> np.ndarray:
    """Plain softmax attention of one query row over [T][d] keys / values."""
    logits = (keys @ q) * scale
    logits = logits - logits.max()
    p = np.exp(logits)
    p /= p.sum()
    return p @ values


def decode(q: np.ndarray, k: np.ndarray, v: np.ndarray, hist_end: int, rk: np.ndarray, rv: np.ndarray,
           tau_k: np.ndarray, tau_v: np.ndarray, scale: float | None = None,
           identity_quantizer: bool = False, heads=None, group: int = 128) -> np.ndarray:
    """Decode output [H_q][d] float64 of one request.

    q [H_q][d], k / v [T][H_kv][d] (float64 holding bf16 values), rk / rv
    [H_kv][d][d] (float64 holding fp32 values), tau_k / tau_v [H_kv].
    ``heads`` restricts the computation to some query heads (others are 0).
    """
    hq, d = q.shape
    hkv = k.shape[1]
    g = hq // hkv
    if scale is None or scale == 0:
        scale = 1.0 / np.sqrt(d)
    out = np.zeros((hq, d))
    want = range(hq) if heads is None else heads
    kv_needed = sorted({h // g for h in want})
    for kvh in kv_needed:
        kt, vt = reconstruct_head(k[:, kvh], v[:, kvh], hist_end, rk[kvh], rv[kvh],
                                  float(tau_k[kvh]), float(tau_v[kvh]), identity_quantizer, group)
        for h in want:
            if h // g == kvh:
                out[h] = softmax_attention(q[h], kt, vt, scale)
    return out


def decode_naive(q, k, v, hist_end, rk, rv, tau_k, tau_v, scale=None, group=128):
    """Per-token loop version of ``decode`` for tiny inputs."""
    hq, d = q.shape
    hkv = k.shape[1]
    g = hq // hkv
    if scale is None or scale == 0:
        scale = 1.0 / np.sqrt(d)
    total = k.shape[0]
    out = np.zeros((hq, d))
    for h in range(hq):
        kvh = h // g
        logits = []
        vals = []
        for j in range(total):
            if SINK <= j < hist_end:
                ck, sk, zk, _ = quant.quantize_tokens(k[j:j + 1, kvh], rk[kvh], np.float32(tau_k[kvh]), group)
                cv, sv, zv, _ = quant.quantize_tokens(v[j:j + 1, kvh], rv[kvh], np.float32(tau_v[kvh]), group)
                sk, zk, sv, zv = (np.reshape(a, (1, -1)) for a in (sk, zk, sv, zv))
                kj = np.zeros(d)
                vj = np.zeros(d)
                for a in range(d):
                    gi = a // group
                    xk = float(zk[0, gi]) + float(sk[0, gi]) * float(ck[0, a])
                    xv = float(zv[0, gi]) + float(sv[0, gi]) * float(cv[0, a])
                    for b in range(d):
                        kj[b] += xk * rk[kvh][b, a]
                        vj[b] += xv * rv[kvh][b, a]
            else:
                kj = k[j, kvh]
                vj = v[j, kvh]
            logits.append(scale * float(np.dot(q[h], kj)))
            vals.append(vj)
        m = max(logits)
        w = [np.exp(x - m) for x in logits]
        tot = sum(w)
        for j in range(total):
            out[h] += (w[j] / tot) * vals[j]
    return out
