"""Offline calibration: per-layer, per-kv-head R_K, R_V and clip thresholds.

This is the one-time offline pass of the pages ("Together AI Open-Sources
OSCAR" (MarkTechPost), Visual Explainer step "Run Offline Calibration"; section
"What OSCAR Does Differently"): estimate the query covariance C_Q and the
score-weighted value covariance C_S from calibration activations, take their
eigenbases U_Q, U_S, and compose R_K = U_Q H_Had P_br, R_V = U_S H_Had P_br;
the clip thresholds are percentiles of the rotated calibration activations.
Its output plays the role of the pages' pre-computed rotation files: fixed
fp32 parameters handed to ``oscar_cache_create``.  It runs once, on the host,
before any decoding -- it is not part of the GPU hot path.

Conventions (shared with every consumer of the rotation files): one R per
(layer, kv head); C_Q pools the query heads of the GQA group; S is the causal
softmax of Q K^T / sqrt(d); eigenvectors by descending eigenvalue with each
column's largest-magnitude entry positive; H_Had = Sylvester order-d Hadamard /
sqrt(d); P_br = bit-reversal of the channel index; tau = ratio-quantile
('linear') of |X R| over all calibration tokens and channels.
"""
from __future__ import annotations

import numpy as np

from . import synth


def walsh_hadamard(d: int) -> np.ndarray:
    h = np.array([[1.0]])
    base = np.array([[1.0, 1.0], [1.0, -1.0]])
    while h.shape[0] < d:
        h = np.kron(base, h)
    return h / np.sqrt(d)


def bit_reverse_indices(d: int) -> np.ndarray:
    bits = d.bit_length() - 1
    return np.array([int(format(i, f"0{bits}b")[::-1], 2) for i in range(d)], dtype=np.int64)


def descending_eigenbasis(c: np.ndarray) -> np.ndarray:
    w, u = np.linalg.eigh(c)
    u = u[:, np.argsort(-w, kind="stable")]
    rows = np.abs(u).argmax(axis=0)
    signs = np.sign(u[rows, np.arange(u.shape[1])])
    return u * np.where(signs == 0, 1.0, signs)


def composed_rotation(u: np.ndarray, bit_reversal: bool = True) -> np.ndarray:
    r = u @ walsh_hadamard(u.shape[0])
    if bit_reversal:
        r = r[:, bit_reverse_indices(u.shape[0])]
    return r


def head_rotations(q_group: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float):
    """(U_Q, U_S) of one kv head from q_group [N][G][d], k, v [N][d] (float64)."""
    n, g, d = q_group.shape
    cq = np.einsum("ngi,ngj->ij", q_group, q_group) / (g * n)
    causal = np.tril(np.ones((n, n), dtype=bool))
    cs = np.zeros((d, d))
    for h in range(g):
        a = np.where(causal, (q_group[:, h] @ k.T) * scale, -np.inf)
        a = np.exp(a - a.max(axis=1, keepdims=True))
        a /= a.sum(axis=1, keepdims=True)
        sv = a @ v
        cs += sv.T @ sv
    cs /= g * n
    return descending_eigenbasis(cq), descending_eigenbasis(cs)


def calibrate_layer(q_cal: np.ndarray, k_cal: np.ndarray, v_cal: np.ndarray, clip_k: float, clip_v: float,
                    bit_reversal: bool = True):
    """fp32 (R_K, R_V) [H_kv][d][d] and fp32 (tau_K, tau_V) [H_kv] of one layer."""
    n, hq, d = q_cal.shape
    hkv = k_cal.shape[1]
    g = hq // hkv
    scale = 1.0 / np.sqrt(d)
    rk = np.empty((hkv, d, d), dtype=np.float32)
    rv = np.empty((hkv, d, d), dtype=np.float32)
    tk = np.empty(hkv, dtype=np.float32)
    tv = np.empty(hkv, dtype=np.float32)
    for h in range(hkv):
        uq, us = head_rotations(q_cal[:, h * g:(h + 1) * g], k_cal[:, h], v_cal[:, h], scale)
        rk[h] = composed_rotation(uq, bit_reversal).astype(np.float32)
        rv[h] = composed_rotation(us, bit_reversal).astype(np.float32)
        tk[h] = np.float32(np.quantile(np.abs(k_cal[:, h] @ rk[h].astype(np.float64)), clip_k, method="linear"))
        tv[h] = np.float32(np.quantile(np.abs(v_cal[:, h] @ rv[h].astype(np.float64)), clip_v, method="linear"))
    return rk, rv, tk, tv


def calibrate_model(cfg_id: int, num_layers: int, num_q_heads: int, num_kv_heads: int, clip_k: float = 0.9,
                    clip_v: float = 0.9, n_cal: int = 512, drift: bool = False, layers=None):
    """Rotation artefacts of a synthetic model: fp32 [L][H_kv][d][d] x2, [L][H_kv] x2.

    ``layers`` limits the fit to some layers (to bound set-up time); every
    other layer then reuses the fit of the first listed layer.
    """
    d = synth.HEAD_DIM
    rk = np.empty((num_layers, num_kv_heads, d, d), dtype=np.float32)
    rv = np.empty_like(rk)
    tk = np.empty((num_layers, num_kv_heads), dtype=np.float32)
    tv = np.empty_like(tk)
    fit = list(range(num_layers)) if layers is None else list(layers)
    for layer in fit:
        q, k, v = synth.calibration_set(cfg_id, layer, num_q_heads, num_kv_heads, n_cal, drift)
        rk[layer], rv[layer], tk[layer], tv[layer] = calibrate_layer(q, k, v, clip_k, clip_v)
    for layer in range(num_layers):
        if layer not in fit:
            rk[layer], rv[layer], tk[layer], tv[layer] = rk[fit[0]], rv[fit[0]], tk[fit[0]], tv[fit[0]]
    return rk, rv, tk, tv
