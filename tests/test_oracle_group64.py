"""Pins of the oracle's G_K = 64 quantiser and record layout.

"Together AI Open-Sources OSCAR" (MarkTechPost), section "What OSCAR Does
Differently": per-token asymmetric INT2 with a default group of G_K = 64
channels, i.e. two groups per 128-channel token-head, each with its own fp16
scale and zero; the same page names the permuted bit-reversal P_br as what
spreads every importance level over the groups, which only matters once a
token-head holds more than one group.  These tests fix the per-group reading
with closed forms, brute force, the byte layout and the 2.5-bit budget.
"""
import numpy as np

from oracle import attention, layout, quant, rotation


def test_closed_form_two_groups():
    # group 0: levels -1.5 .. 1.5 (s = 1), group 1: ten times wider (s = 10, z = -15)
    x = np.array([(j % 4) - 1.5 for j in range(64)] + [10 * ((j % 4) - 1.5) for j in range(64)], np.float32)
    c, s, z = quant.quantize_groups(x[None], np.float32(100.0), group=64)
    assert s.shape == (1, 2) and z.shape == (1, 2)
    assert [float(v) for v in s[0]] == [1.0, 10.0] and [float(v) for v in z[0]] == [-1.5, -15.0]
    assert np.array_equal(c[0], np.arange(128) % 4)
    xh = quant.dequantize(c, s, z)
    assert np.array_equal(xh[0], x.astype(np.float64))


def test_groups_are_independent():
    # changing group 1 never changes group 0's codes or meta, and vice versa
    rng = np.random.default_rng(0)
    x = (rng.standard_normal((50, 128)) * 2).astype(np.float32)
    y = x.copy()
    y[:, 64:] = (rng.standard_normal((50, 64)) * 7).astype(np.float32)
    tau = np.float32(5.0)
    cx, sx, zx = quant.quantize_groups(x, tau, group=64)
    cy, sy, zy = quant.quantize_groups(y, tau, group=64)
    assert np.array_equal(cx[:, :64], cy[:, :64])
    assert np.array_equal(sx[:, 0].view(np.uint16), sy[:, 0].view(np.uint16))
    assert np.array_equal(zx[:, 0].view(np.uint16), zy[:, 0].view(np.uint16))
    assert not np.array_equal(sx[:, 1], sy[:, 1])


def test_nearest_level_brute_force_per_group():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((300, 128)) * rng.uniform(0.1, 10, (300, 1))).astype(np.float32)
    x[:, 64:] *= 3.0
    tau = np.float32(12.0)
    c, s, z = quant.quantize_groups(x, tau, group=64)
    t = quant.t_values(x, tau, s, z)
    xc = np.clip(x.astype(np.float64), -12.0, 12.0)
    for g in range(2):
        sl = slice(64 * g, 64 * g + 64)
        levels = z[:, g].astype(np.float64)[:, None, None] + \
            s[:, g].astype(np.float64)[:, None, None] * np.arange(4)[None, None, :]
        best = np.abs(xc[:, sl, None] - levels).argmin(axis=-1)
        near_tie = np.abs(t[:, sl] - np.round(t[:, sl] - 0.5) - 0.5) < 1e-5
        assert not ((best != c[:, sl]) & ~near_tie).any()
        # each group's zero is its own clipped minimum, rounded to fp16
        assert np.array_equal(z[:, g].view(np.uint16),
                              xc[:, sl].min(axis=1).astype(np.float32).astype(np.float16).view(np.uint16))


def test_finer_groups_never_widen_the_scale():
    # a group's range is inside the token-head's range, so s_64 <= s_128 for each group
    rng = np.random.default_rng(2)
    x = (rng.standard_normal((400, 128)) * rng.uniform(0.1, 4, (400, 1))).astype(np.float32)
    tau = np.float32(3.0)
    _, s128, _ = quant.quantize_groups(x, tau)
    _, s64, _ = quant.quantize_groups(x, tau, group=64)
    assert np.all(s64.astype(np.float64) <= s128.astype(np.float64)[:, None])


def test_record_layout_and_bits():
    lay = layout.record_layout(64)
    assert (lay["k_meta"], lay["v_meta"], lay["meta_bytes"], lay["record"]) == (4096, 4608, 8, 5120)
    assert lay["record"] == 64 * 80                         # 80 B per token-head
    assert 8 * 80 / 128 == 5.0                              # K and V: 2.5 bits per element each
    assert layout.record_layout(128)["record"] == layout.RECORD_BYTES == 4608
    # long-context average: the INT2 share dominates, 2.5 bits plus the BF16 windows
    assert abs(layout.bits_per_element(10 ** 7, group=64) - 2.5) < 1e-3
    assert abs(layout.bits_per_element(10 ** 7) - 2.25) < 1e-3


def test_meta_bytes_two_groups_roundtrip():
    s = np.array([[1.0, 0.5], [2.0, 65504.0]], dtype=np.float16)
    z = np.array([[-1.5, 0.25], [-0.0, 2.0 ** -24]], dtype=np.float16)
    m = layout.meta_bytes(s, z, groups=2)
    assert m.shape == (2, 8)
    assert list(m[0]) == [0x00, 0x3C, 0x00, 0xBE, 0x00, 0x38, 0x00, 0x34]   # 1, -1.5, 0.5, 0.25
    s2, z2 = layout.meta_to_sz(m)
    assert np.array_equal(s2.view(np.uint16), s.view(np.uint16))
    assert np.array_equal(z2.view(np.uint16), z.view(np.uint16))


def test_channel_permutation_matters_only_with_two_groups():
    # one group: permuting channels permutes the codes and keeps (s, z); two groups:
    # the bit-reversal sends half of each group to the other one, and (s, z) change
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((64, 128)) * np.linspace(0.2, 5.0, 128)).astype(np.float32)
    pi = rotation.bit_reversal(128)
    tau = np.float32(100.0)
    c, s, z = quant.quantize_groups(x, tau)
    cp, sp, zp = quant.quantize_groups(x[:, pi], tau)
    assert np.array_equal(cp, c[:, pi]) and np.array_equal(sp, s) and np.array_equal(zp, z)
    _, s2, _ = quant.quantize_groups(x, tau, group=64)
    _, s2p, _ = quant.quantize_groups(x[:, pi], tau, group=64)
    assert not np.array_equal(s2, s2p)
    # the bit-reversal interleaves: each group of the permuted row takes every other channel
    assert sorted(pi[:64] % 2) == [0] * 64 and sorted(pi[64:] % 2) == [1] * 64


def test_decode_naive_matches_vectorised_at_group64():
    rng = np.random.default_rng(4)
    T, hkv, hq, d = 72, 1, 2, 128
    k = rng.standard_normal((T, hkv, d)).astype(np.float32).astype(np.float64)
    v = rng.standard_normal((T, hkv, d)).astype(np.float32).astype(np.float64)
    q = rng.standard_normal((hq, d))
    r = np.linalg.qr(rng.standard_normal((d, d)))[0].astype(np.float32).astype(np.float64)
    rk = rv = r[None]
    tk = tv = np.array([2.5], np.float32)
    a = attention.decode(q, k, v, 70, rk, rv, tk, tv, group=64)
    b = attention.decode_naive(q, k, v, 70, rk, rv, tk, tv, group=64)
    assert np.max(np.abs(a - b)) < 1e-12
    # and it differs from the 128-group decode (the meta really is per group)
    c = attention.decode(q, k, v, 70, rk, rv, tk, tv)
    assert np.max(np.abs(a - c)) > 1e-6
