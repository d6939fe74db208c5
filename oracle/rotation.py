"""Offline rotation construction (oracle; test infrastructure).

[MTP] section "What OSCAR Does Differently":
  * key error in the logits is weighted by the query covariance
    C_Q = (1/N) sum_n q_n^T q_n; U_Q are its eigenvectors;
  * value error is weighted by the score-weighted value covariance
    C_S = (1/N) V^T S^T S V; U_S are its eigenvectors;
  * R_K = U_Q . H_Had . P_br and R_V = U_S . H_Had . P_br;
  * Lemma 1: every diagonal entry of H_Had^T Lambda H_Had equals tr(Lambda)/d;
  * P_br is a bit-reversal permutation of the channels.
[MS] section "OSCAR的设计": one fixed rotation and clip threshold per layer and
head; R = U . Hadamard . bit-reversal.

Readings where the pages are silent:
  * one R per (layer, kv-head); C_Q pools the query heads of the kv-head's GQA
    group; S is the causal softmax of Q K^T / sqrt(128) over the calibration
    tokens;
  * eigenvectors sorted by descending eigenvalue; each column's
    largest-magnitude entry made positive (first such entry on ties);
  * H_Had is the Sylvester Hadamard matrix scaled by 1/sqrt(128), natural order;
  * clip threshold tau = the c-quantile (numpy 'linear' method) of |X R| over
    all calibration tokens and channels, stored as fp32.
Parity of the calibration recipe itself is unpinned by the pages (no worked
values); the pieces are pinned by the orthogonality, involution, Lemma-1 and
logit-error identities.
"""
from __future__ import annotations

import numpy as np


def sylvester_hadamard(n: int = 128) -> np.ndarray:
    """Orthonormal Walsh-Hadamard matrix of order n (a power of two), float64."""
    h = np.ones((1, 1))
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    assert h.shape[0] == n, "order must be a power of two"
    return h / np.sqrt(n)


def bit_reversal(n: int = 128) -> np.ndarray:
    """pi[i] = i with its log2(n) bits reversed."""
    bits = n.bit_length() - 1
    assert 1 << bits == n
    out = np.zeros(n, dtype=np.int64)
    for i in range(n):
        r = 0
        for b in range(bits):
            if i >> b & 1:
                r |= 1 << (bits - 1 - b)
        out[i] = r
    return out


def permutation_matrix(pi: np.ndarray) -> np.ndarray:
    """P with (M P)[:, j] = M[:, pi[j]]."""
    n = len(pi)
    p = np.zeros((n, n))
    for j in range(n):
        p[pi[j], j] = 1.0
    return p


def sorted_eigenvectors(c: np.ndarray) -> np.ndarray:
    """Columns = eigenvectors of symmetric c by descending eigenvalue, sign-fixed."""
    w, u = np.linalg.eigh(c)
    order = np.argsort(-w, kind="stable")
    u = u[:, order].copy()
    for j in range(u.shape[1]):
        i = int(np.argmax(np.abs(u[:, j])))
        if u[i, j] < 0:
            u[:, j] = -u[:, j]
    return u


def query_covariance(q_group: np.ndarray) -> np.ndarray:
    """C_Q = (1/(G N)) sum over the group's heads and tokens of q^T q.

    q_group: [N][G][d] calibration queries of the G query heads of one kv-head.
    """
    n, g, d = q_group.shape
    c = np.zeros((d, d))
    for h in range(g):
        qh = q_group[:, h, :]
        c += qh.T @ qh
    return c / (g * n)


def causal_softmax_scores(q: np.ndarray, k: np.ndarray, scale: float) -> np.ndarray:
    """S[n, m] = softmax over m <= n of scale * q_n . k_m (0 for m > n)."""
    logits = (q @ k.T) * scale
    n = logits.shape[0]
    mask = np.tril(np.ones((n, n), dtype=bool))
    logits = np.where(mask, logits, -np.inf)
    logits -= logits.max(axis=1, keepdims=True)
    e = np.exp(logits)
    return e / e.sum(axis=1, keepdims=True)


def score_weighted_value_covariance(q_group: np.ndarray, k: np.ndarray, v: np.ndarray,
                                    scale: float) -> np.ndarray:
    """C_S = (1/(G N)) sum_g V^T S_g^T S_g V over the group's query heads."""
    n, g, d = q_group.shape
    c = np.zeros((d, d))
    for h in range(g):
        s = causal_softmax_scores(q_group[:, h, :], k, scale)
        sv = s @ v
        c += sv.T @ sv
    return c / (g * n)


def compose_rotation(u: np.ndarray, use_bit_reversal: bool = True) -> np.ndarray:
    """R = U . H_Had . P_br (float64)."""
    d = u.shape[0]
    r = u @ sylvester_hadamard(d)
    if use_bit_reversal:
        r = r @ permutation_matrix(bit_reversal(d))
    return r


def clip_threshold(x_rot: np.ndarray, ratio: float) -> float:
    """tau = ratio-quantile of |x_rot| over all tokens and channels, as fp32."""
    return float(np.float32(np.quantile(np.abs(x_rot).ravel(), ratio, method="linear")))


def build_layer_rotations(q_cal: np.ndarray, k_cal: np.ndarray, v_cal: np.ndarray,
                          clip_k: float, clip_v: float, use_bit_reversal: bool = True):
    """Per-kv-head rotations and thresholds of one layer.

    q_cal [N][H_q][d], k_cal / v_cal [N][H_kv][d] (float64, bf16-valued).
    Returns (R_K, R_V) float64 [H_kv][d][d] before fp32 rounding, and
    (tau_K, tau_V) fp32 [H_kv] computed with the fp32-rounded rotations.
    """
    n, hq, d = q_cal.shape
    hkv = k_cal.shape[1]
    g = hq // hkv
    scale = 1.0 / np.sqrt(d)
    rk = np.zeros((hkv, d, d))
    rv = np.zeros((hkv, d, d))
    tk = np.zeros(hkv, dtype=np.float32)
    tv = np.zeros(hkv, dtype=np.float32)
    for h in range(hkv):
        qg = q_cal[:, h * g:(h + 1) * g, :]
        uq = sorted_eigenvectors(query_covariance(qg))
        us = sorted_eigenvectors(score_weighted_value_covariance(qg, k_cal[:, h], v_cal[:, h], scale))
        rk[h] = compose_rotation(uq, use_bit_reversal)
        rv[h] = compose_rotation(us, use_bit_reversal)
        rk32 = rk[h].astype(np.float32).astype(np.float64)
        rv32 = rv[h].astype(np.float32).astype(np.float64)
        tk[h] = clip_threshold(k_cal[:, h] @ rk32, clip_k)
        tv[h] = clip_threshold(v_cal[:, h] @ rv32, clip_v)
    return rk, rv, tk, tv
