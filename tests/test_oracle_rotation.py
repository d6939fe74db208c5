"""Pins of the oracle's rotation construction against closed forms and identities.

[MTP] = "Together AI Open-Sources OSCAR" (MarkTechPost), section "What OSCAR
Does Differently": logit-error identity, C_Q, C_S, R = U . H_Had . P_br,
Lemma 1, bit reversal.
"""
import numpy as np
import pytest

from oracle import attention, quant, rotation


def test_hadamard_closed_form():
    h = rotation.sylvester_hadamard(128)
    assert np.allclose(np.abs(h), 1 / np.sqrt(128), atol=0, rtol=1e-15)
    assert np.abs(h @ h - np.eye(128)).max() < 1e-12          # symmetric and orthonormal: H^2 = I
    assert np.all(h[0] > 0) and np.all(h[:, 0] > 0)           # Sylvester natural order
    # row i, column j sign = (-1)^popcount(i & j)
    for i, j in [(1, 1), (3, 5), (127, 127), (64, 65), (77, 12)]:
        assert np.sign(h[i, j]) == (-1) ** bin(i & j).count("1")


def test_bit_reversal_values_and_involution():
    pi = rotation.bit_reversal(128)
    assert pi[0] == 0 and pi[1] == 64 and pi[2] == 32 and pi[3] == 96 and pi[127] == 127 and pi[6] == 48
    assert np.array_equal(pi[pi], np.arange(128))
    p = rotation.permutation_matrix(pi)
    assert np.array_equal(p @ p, np.eye(128))
    m = np.arange(128 * 128, dtype=float).reshape(128, 128)
    assert np.array_equal((m @ p)[:, 1], m[:, 64])


def test_lemma1_equal_channel_importance():
    rng = np.random.default_rng(0)
    h = rotation.sylvester_hadamard(128)
    lam = np.diag(rng.exponential(size=128) ** 3)             # a peaky spectrum
    d = np.diag(h.T @ lam @ h)
    assert np.abs(d - np.trace(lam) / 128).max() < 1e-12


def test_lemma1_after_covariance_diagonalisation():
    rng = np.random.default_rng(1)
    a = rng.standard_normal((128, 128)) * np.linspace(0.1, 5, 128)
    c = a @ a.T
    u = rotation.sorted_eigenvectors(c)
    r = rotation.compose_rotation(u)
    d = np.diag(r.T @ c @ r)
    assert np.abs(d - np.trace(c) / 128).max() < 1e-9 * np.trace(c)


def test_sorted_eigenvectors_closed_form():
    c = np.diag([1.0, 5.0, 3.0, 0.5])
    u = rotation.sorted_eigenvectors(c)
    expect = np.zeros((4, 4))
    expect[1, 0] = expect[2, 1] = expect[0, 2] = expect[3, 3] = 1.0
    assert np.array_equal(u, expect)


def test_query_covariance_normalisation():
    q = np.zeros((2, 1, 4))
    q[0, 0, 0] = 1.0
    q[1, 0, 1] = 2.0
    assert np.array_equal(rotation.query_covariance(q), np.diag([0.5, 2.0, 0.0, 0.0]))
    # pooling over a GQA group divides by G * N
    q2 = np.concatenate([q, q], axis=1)
    assert np.array_equal(rotation.query_covariance(q2), np.diag([0.5, 2.0, 0.0, 0.0]))


def test_score_weighted_covariance_matches_attention_outputs():
    rng = np.random.default_rng(2)
    n, d = 12, 128
    q = rng.standard_normal((n, 1, d))
    k = rng.standard_normal((n, d))
    v = rng.standard_normal((n, d))
    scale = 1 / np.sqrt(d)
    c = rotation.score_weighted_value_covariance(q, k, v, scale)
    # each row of S V is a causal attention output; C_S is the mean outer product
    rows = np.array([attention.softmax_attention(q[i, 0], k[:i + 1], v[:i + 1], scale) for i in range(n)])
    ref = sum(np.outer(x, x) for x in rows) / n
    assert np.abs(c - ref).max() < 1e-12


def test_score_weighted_covariance_constant_values():
    rng = np.random.default_rng(3)
    n, d = 9, 128
    vrow = rng.standard_normal(d)
    c = rotation.score_weighted_value_covariance(rng.standard_normal((n, 2, d)), rng.standard_normal((n, d)),
                                                 np.tile(vrow, (n, 1)), 0.1)
    assert np.abs(c - np.outer(vrow, vrow)).max() < 1e-12


def _layer(seed=0, g=4):
    rng = np.random.default_rng(seed)
    n, d = 256, 128
    q = rng.standard_normal((n, g, d)) @ rng.standard_normal((d, d)) / np.sqrt(d)
    k = rng.standard_normal((n, 1, d))
    k[..., :4] *= 20
    v = rng.standard_normal((n, 1, d))
    v[..., 5:9] *= 20
    return q, k, v


def test_built_rotation_orthogonal():
    q, k, v = _layer()
    rk, rv, tk, tv = rotation.build_layer_rotations(q, k, v, 0.9, 0.9)
    for r in (rk[0], rv[0]):
        assert np.abs(r.T @ r - np.eye(128)).max() < 1e-12
    assert tk[0] > 0 and tv[0] > 0
    # tau is the 0.9-quantile: ~10 % of |rotated| calibration values exceed it
    xr = k[:, 0] @ rk[0].astype(np.float32).astype(np.float64)
    frac = np.mean(np.abs(xr) > tk[0])
    assert 0.095 < frac < 0.105


def test_logit_error_identity():
    """The identity |Q K^T - Q K^^T|_F^2 = tr((K - K^) Q^T Q (K - K^)^T) that "Together AI
    Open-Sources OSCAR" (MarkTechPost), section "What OSCAR Does Differently", builds its
    objective on.  It holds for any K^, so this checks the page's argument; it pins
    nothing of the oracle."""
    rng = np.random.default_rng(4)
    q = rng.standard_normal((64, 128))
    k = rng.standard_normal((300, 128))
    khat = k + 0.01 * rng.standard_normal(k.shape)
    lhs = np.linalg.norm(q @ k.T - q @ khat.T) ** 2
    e = k - khat
    rhs = np.trace(e @ q.T @ q @ e.T)
    assert abs(lhs - rhs) <= 1e-9 * lhs


def test_logit_error_identity_with_oracle_quantiser():
    """The same identity with K^ from the oracle's quantiser: a check of the page's
    identity (true for any K^), not a pin of the quantiser, which the brute-force and
    closed-form tests in test_oracle_quant.py pin."""
    q, k, v = _layer(5)
    rk, rv, tk, tv = rotation.build_layer_rotations(q, k, v, 0.9, 0.9)
    rk32 = rk[0].astype(np.float32).astype(np.float64)
    toks = k[:, 0]
    c, s, z, _ = quant.quantize_tokens(toks, rk32, tk[0])
    khat = quant.dequantize(c, s, z) @ rk32.T
    qq = q[:, 0, :]
    lhs = np.linalg.norm(qq @ toks.T - qq @ khat.T) ** 2
    e = toks - khat
    rhs = np.trace(e @ qq.T @ qq @ e.T)
    assert abs(lhs - rhs) <= 1e-9 * lhs


def test_bit_reversal_invariance_at_group_128():
    """With one group of 128 channels, P_br only relabels channels inside the group."""
    q, k, v = _layer(6)
    n, g, d = q.shape
    u = rotation.sorted_eigenvectors(rotation.query_covariance(q))
    r1 = rotation.compose_rotation(u, True).astype(np.float32).astype(np.float64)
    r0 = rotation.compose_rotation(u, False).astype(np.float32).astype(np.float64)
    tau = np.float32(3.0)
    c1, s1, z1, _ = quant.quantize_tokens(k[:, 0], r1, tau)
    c0, s0, z0, _ = quant.quantize_tokens(k[:, 0], r0, tau)
    assert np.array_equal(s1, s0) and np.array_equal(z1, z0)
    k1 = quant.dequantize(c1, s1, z1) @ r1.T
    k0 = quant.dequantize(c0, s0, z0) @ r0.T
    assert np.abs(k1 - k0).max() < 1e-12


@pytest.mark.parametrize("plant", ["drop_hadamard_scale", "ascending_eigs"])
def test_planted_mistakes_are_caught(plant, monkeypatch):
    """A plausible slip in the rotation builder breaks one of the pins above."""
    if plant == "drop_hadamard_scale":
        orig = rotation.sylvester_hadamard
        monkeypatch.setattr(rotation, "sylvester_hadamard", lambda n=128: orig(n) * np.sqrt(n))
        with pytest.raises(AssertionError):
            test_built_rotation_orthogonal()
    else:
        def ascending(c):
            w, u = np.linalg.eigh(c)
            return u
        monkeypatch.setattr(rotation, "sorted_eigenvectors", ascending)
        with pytest.raises(AssertionError):
            test_sorted_eigenvectors_closed_form()
