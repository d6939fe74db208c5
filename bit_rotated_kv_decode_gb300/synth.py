"""Seeded synthetic inputs shared by the CUDA path and the oracle.

This module only draws random numbers.  It holds none of the method's
arithmetic (no rotation, clipping, quantisation, packing or attention), so
both sides of every parity check can take their inputs from here without
sharing any of the computation under test.

Workloads follow the shapes of the Qwen3 attention layers the pages evaluate
(head_dim 128, 8 KV heads, 32 or 64 query heads) at 2K-128K contexts:

* K and V: bf16 drawn from N(0, 1); per (layer, kv-head) four fixed channels,
  chosen without replacement separately for K and for V, are scaled by 20 to
  model channel-wise outliers ("Together AI Open-Sources OSCAR", MarkTechPost,
  section "Why INT2 KV Cache Quantization is Hard").
* q: drawn from N(0, Sigma) with Sigma = A A^T / 128, A a seeded 128x128
  Gaussian per (layer, query head).
* An optional slow drift of the channel means for the 128K workload:
  mu_c(t) = mu0_c + (t / T) * delta_c with mu0, delta ~ N(0, 0.5^2).
* Calibration sets of 512 tokens per head drawn from the same laws.
* A second law for the rotation ablation, a shared low-rank subspace: per
  (layer, kv head) a seeded orthonormal basis u_1..u_4 of a 4-dimensional
  subspace; keys k = x + 6 sum_i z_i u_i (x ~ N(0, 1) with the four outlier
  channels scaled by 5 instead of 20, z ~ N(0, 1)); values alike with a basis
  of their own; the group's queries q = 3 sum_i z_i u_i + 0.3 N(0, I).  Queries
  then have a few dominant eigen-directions, which keys share ("Together AI
  Open-Sources OSCAR", MarkTechPost, section "What OSCAR Does Differently":
  the rotation is aligned with the query covariance's dominant directions).

Seeds: seed(cfg, layer, head, purpose) = splitmix64(cfg<<40 | layer<<24 |
head<<8 | purpose).  Tensors are drawn with torch generators on the device
they are requested on; a CPU draw and a CUDA draw of the same seed differ, so
a parity check always feeds both sides from the same drawn tensor.
"""
from __future__ import annotations

import numpy as np
import torch

MASK64 = (1 << 64) - 1

# purpose ids of the seed derivation
P_OUTLIER_K = 1
P_OUTLIER_V = 2
P_K = 3
P_V = 4
P_QMIX = 5
P_Q = 6
P_CAL_K = 7
P_CAL_V = 8
P_CAL_Q = 9
P_DRIFT_K = 10
P_DRIFT_V = 11
P_APPEND_K = 12
P_APPEND_V = 13
P_LENGTHS = 14
P_PREFIX_K = 15
P_PREFIX_V = 16
P_SUB_BASIS_K = 17
P_SUB_BASIS_V = 18
P_SUB_Z = 19

OUTLIER_CHANNELS = 4
OUTLIER_SCALE = 20.0
HEAD_DIM = 128


def splitmix64(x: int) -> int:
    """One output of SplitMix64 (Steele, Lea, Flood 2014) for state ``x``."""
    z = (x + 0x9E3779B97F4A7C15) & MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def seed_for(cfg: int, layer: int, head: int, purpose: int, step: int = 0) -> int:
    """Seed of one draw; ``step`` separates draws repeated per decode step."""
    key = ((cfg << 40) | (layer << 24) | (head << 8) | purpose) & MASK64
    s = splitmix64(key)
    if step:
        s = splitmix64(s ^ (step & MASK64))
    return s & ((1 << 63) - 1)


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def outlier_channels(cfg: int, layer: int, num_kv_heads: int, which: str) -> np.ndarray:
    """int64 [H_kv][4]: the outlier channels of K (``which='k'``) or V."""
    purpose = P_OUTLIER_K if which == "k" else P_OUTLIER_V
    out = np.empty((num_kv_heads, OUTLIER_CHANNELS), dtype=np.int64)
    for h in range(num_kv_heads):
        rng = np.random.Generator(np.random.PCG64(seed_for(cfg, layer, h, purpose)))
        out[h] = rng.choice(HEAD_DIM, OUTLIER_CHANNELS, replace=False)
    return out


def channel_scale(cfg: int, layer: int, num_kv_heads: int, which: str) -> np.ndarray:
    """float32 [H_kv][128]: 1 everywhere, 20 on the outlier channels."""
    sc = np.ones((num_kv_heads, HEAD_DIM), dtype=np.float32)
    ch = outlier_channels(cfg, layer, num_kv_heads, which)
    for h in range(num_kv_heads):
        sc[h, ch[h]] = OUTLIER_SCALE
    return sc


def drift_params(cfg: int, layer: int, num_kv_heads: int, which: str):
    """(mu0, delta), float32 [H_kv][128] each, drawn from N(0, 0.5^2)."""
    purpose = P_DRIFT_K if which == "k" else P_DRIFT_V
    rng = np.random.Generator(np.random.PCG64(seed_for(cfg, layer, 0, purpose)))
    mu0 = rng.normal(0.0, 0.5, size=(num_kv_heads, HEAD_DIM)).astype(np.float32)
    delta = rng.normal(0.0, 0.5, size=(num_kv_heads, HEAD_DIM)).astype(np.float32)
    return mu0, delta


def kv_tokens(cfg: int, layer: int, num_kv_heads: int, which: str, positions: torch.Tensor | range,
              total_len: int = 0, drift: bool = False, device="cpu", purpose: int | None = None,
              stream_id: int = 0) -> torch.Tensor:
    """bf16 [n][H_kv][128] K or V rows for the given token positions.

    Rows are drawn in one block for the whole ``positions`` range (which must
    be contiguous), so one call per (layer, which, stream_id) defines the data.
    ``stream_id`` separates independent sequences (requests, appended tokens).
    """
    if isinstance(positions, range):
        p0, n = positions.start, len(positions)
    else:
        p0, n = int(positions[0]), int(positions.numel())
    if purpose is None:
        purpose = P_K if which == "k" else P_V
    g = _gen(device, seed_for(cfg, layer, stream_id, purpose, step=p0 + 1))
    x = torch.randn((n, num_kv_heads, HEAD_DIM), generator=g, device=device, dtype=torch.float32)
    sc = torch.from_numpy(channel_scale(cfg, layer, num_kv_heads, which)).to(device)
    x.mul_(sc)
    if drift:
        mu0, delta = drift_params(cfg, layer, num_kv_heads, which)
        t = torch.arange(p0, p0 + n, device=device, dtype=torch.float32) / float(max(total_len, 1))
        x.add_(torch.from_numpy(mu0).to(device)[None])
        x.add_(t[:, None, None] * torch.from_numpy(delta).to(device)[None])
    return x.to(torch.bfloat16)


def query_mix(cfg: int, layer: int, num_q_heads: int, device="cpu") -> torch.Tensor:
    """float32 [H_q][128][128]: the seeded Gaussian A of each query head."""
    g = _gen(device, seed_for(cfg, layer, 0, P_QMIX))
    return torch.randn((num_q_heads, HEAD_DIM, HEAD_DIM), generator=g, device=device, dtype=torch.float32)


def queries(cfg: int, layer: int, num_q_heads: int, n: int, step: int, device="cpu",
            purpose: int = P_Q, mix: torch.Tensor | None = None) -> torch.Tensor:
    """bf16 [n][H_q][128] queries q = z A^T / sqrt(128), z ~ N(0, I)."""
    if mix is None:
        mix = query_mix(cfg, layer, num_q_heads, device)
    g = _gen(device, seed_for(cfg, layer, 0, purpose, step=step + 1))
    z = torch.randn((n, num_q_heads, HEAD_DIM), generator=g, device=device, dtype=torch.float32)
    q = torch.einsum("nhi,hoi->nho", z, mix) / np.sqrt(HEAD_DIM)
    return q.to(torch.bfloat16).contiguous()


def calibration_set(cfg: int, layer: int, num_q_heads: int, num_kv_heads: int, n: int = 512,
                    drift: bool = False):
    """Host float64 calibration tensors (Q [n][H_q][128], K, V [n][H_kv][128]).

    Drawn on the CPU from the same laws as the workload, values rounded to bf16
    like the activations they stand in for.
    """
    k = kv_tokens(cfg, layer, num_kv_heads, "k", range(0, n), total_len=n, drift=drift, purpose=P_CAL_K)
    v = kv_tokens(cfg, layer, num_kv_heads, "v", range(0, n), total_len=n, drift=drift, purpose=P_CAL_V)
    q = queries(cfg, layer, num_q_heads, n, step=0, purpose=P_CAL_Q)
    return (q.to(torch.float64).numpy(), k.to(torch.float64).numpy(), v.to(torch.float64).numpy())


def request_lengths(cfg: int, batch: int, lo: int, hi: int) -> list[int]:
    """Seeded context lengths drawn uniformly from [lo, hi]."""
    rng = np.random.Generator(np.random.PCG64(seed_for(cfg, 0, 0, P_LENGTHS)))
    return [int(x) for x in rng.integers(lo, hi + 1, size=batch)]


# ---- the shared low-rank subspace law of the rotation ablation -------------------------------
SUBSPACE_RANK = 4
SUBSPACE_KV_SCALE = 6.0
SUBSPACE_Q_SCALE = 3.0
SUBSPACE_Q_NOISE = 0.3
SUBSPACE_OUTLIER_SCALE = 5.0


def subspace_basis(cfg: int, layer: int, kv_head: int, which: str) -> np.ndarray:
    """float64 [128][SUBSPACE_RANK]: orthonormal columns u_1..u_r of the head's subspace
    (the Q factor, with a positive R diagonal, of a seeded Gaussian)."""
    purpose = P_SUB_BASIS_K if which == "k" else P_SUB_BASIS_V
    rng = np.random.Generator(np.random.PCG64(seed_for(cfg, layer, kv_head, purpose)))
    a = rng.normal(size=(HEAD_DIM, SUBSPACE_RANK))
    qf, rf = np.linalg.qr(a)
    return qf * np.sign(np.diag(rf))[None, :]


def _subspace_part(cfg, layer, heads, which_basis, n, scale, seed, device):
    """[n][len(heads)][128] float32: scale * sum_i z_i u_i per head, z ~ N(0, 1)."""
    g = _gen(device, seed)
    z = torch.randn((n, len(heads), SUBSPACE_RANK), generator=g, device=device, dtype=torch.float32)
    basis = torch.from_numpy(np.stack([subspace_basis(cfg, layer, h, which_basis) for h in heads])).to(
        device=device, dtype=torch.float32)                       # [heads][128][r]
    return scale * torch.einsum("nhr,hdr->nhd", z, basis)


def subspace_kv(cfg: int, layer: int, num_kv_heads: int, which: str, n: int, device="cpu",
                calibration: bool = False, stream_id: int = 0) -> torch.Tensor:
    """bf16 [n][H_kv][128] K or V rows of the shared-subspace law."""
    if which == "k":
        purpose = P_CAL_K if calibration else P_K
    else:
        purpose = P_CAL_V if calibration else P_V
    g = _gen(device, seed_for(cfg, layer, stream_id, purpose, step=1))
    x = torch.randn((n, num_kv_heads, HEAD_DIM), generator=g, device=device, dtype=torch.float32)
    sc = torch.from_numpy(channel_scale(cfg, layer, num_kv_heads, which)).to(device)
    x.mul_(torch.where(sc > 1.0, torch.full_like(sc, SUBSPACE_OUTLIER_SCALE), sc))
    x.add_(_subspace_part(cfg, layer, range(num_kv_heads), which, n, SUBSPACE_KV_SCALE,
                          seed_for(cfg, layer, stream_id, P_SUB_Z, step=purpose), device))
    return x.to(torch.bfloat16)


def subspace_queries(cfg: int, layer: int, num_q_heads: int, num_kv_heads: int, n: int, step: int,
                     device="cpu", purpose: int = P_Q) -> torch.Tensor:
    """bf16 [n][H_q][128] queries of the shared-subspace law: query head h draws in the
    key subspace of kv head h // (H_q / H_kv)."""
    g_size = num_q_heads // num_kv_heads
    heads = [h // g_size for h in range(num_q_heads)]
    q = _subspace_part(cfg, layer, heads, "k", n, SUBSPACE_Q_SCALE,
                       seed_for(cfg, layer, 0, purpose, step=step + 1), device)
    g = _gen(device, seed_for(cfg, layer, 1, purpose, step=step + 1))
    q.add_(SUBSPACE_Q_NOISE * torch.randn((n, num_q_heads, HEAD_DIM), generator=g, device=device,
                                          dtype=torch.float32))
    return q.to(torch.bfloat16).contiguous()


def subspace_calibration_set(cfg: int, layer: int, num_q_heads: int, num_kv_heads: int, n: int = 512):
    """Host float64 calibration tensors of the shared-subspace law (as calibration_set)."""
    k = subspace_kv(cfg, layer, num_kv_heads, "k", n, calibration=True)
    v = subspace_kv(cfg, layer, num_kv_heads, "v", n, calibration=True)
    q = subspace_queries(cfg, layer, num_q_heads, num_kv_heads, n, 0, purpose=P_CAL_Q)
    return (q.to(torch.float64).numpy(), k.to(torch.float64).numpy(), v.to(torch.float64).numpy())
