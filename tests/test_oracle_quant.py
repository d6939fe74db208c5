"""Pins of the oracle's rotation rounding, INT2 quantiser and packing.

The pages fix: per-token asymmetric INT2 with scale and zero point, groups of
128 channels, four codes per byte ("Together AI Open-Sources OSCAR",
MarkTechPost, section The Serving System; "TogetherAI开源OSCAR", ModelScope,
sections OSCAR的设计 and 快速实践).  The exact convention is a reading; these
tests pin it with closed forms, ties, brute force and error bounds.
"""
from fractions import Fraction

import numpy as np
import pytest

from oracle import layout, quant


def _group(vals):
    x = np.zeros(128, dtype=np.float32)
    x[:len(vals)] = vals
    x[len(vals):] = vals[-1]
    return x


def test_closed_form_four_levels_and_byte_order():
    x = np.array([(j % 4) - 1.5 for j in range(128)], dtype=np.float32)
    c, s, z = quant.quantize_groups(x[None], np.float32(100.0))
    assert float(s[0]) == 1.0 and float(z[0]) == -1.5
    assert np.array_equal(c[0], np.arange(128) % 4)
    packed = layout.pack_codes(c)
    assert np.all(packed == 0xE4)                 # 0 | 1<<2 | 2<<4 | 3<<6
    assert np.array_equal(layout.unpack_codes(packed), c)


def test_record_slot_fields_offsets():
    """A slot's fields sit at 32 r (K codes), 2048 + 32 r (V codes), 4096 + 4 r and
    4352 + 4 r (meta) of a 4608-byte record; with G_K = 64 the meta is 8 bytes per
    slot at 4096 + 8 r and 4608 + 8 r."""
    rec = np.arange(4608, dtype=np.int64).astype(np.uint8)
    kc, vc, km, vm = layout.record_slot_fields(rec, 9)
    assert np.array_equal(kc, rec[288:320]) and np.array_equal(vc, rec[2048 + 288:2048 + 320])
    assert np.array_equal(km, rec[4096 + 36:4096 + 40]) and np.array_equal(vm, rec[4352 + 36:4352 + 40])
    rec64 = np.arange(5120, dtype=np.int64).astype(np.uint8)
    kc, vc, km, vm = layout.record_slot_fields(rec64, 9, group=64)
    assert np.array_equal(km, rec64[4096 + 72:4096 + 80]) and np.array_equal(vm, rec64[4608 + 72:4608 + 80])


def test_round_half_to_even_ties():
    # z = 0, s = 1 -> t = x; ties at 0.5, 1.5, 2.5 go to 0, 2, 2
    x = _group([0.0, 0.5, 1.5, 2.5, 3.0, 0.49, 1.51, 2.2])
    c, s, z = quant.quantize_groups(x[None], np.float32(10.0))
    assert float(s[0]) == 1.0 and float(z[0]) == 0.0
    assert list(c[0, :8]) == [0, 0, 2, 2, 3, 0, 2, 2]


def test_clip_to_threshold():
    x = _group([-5.0, 5.0, 0.25, 0.0])
    c, s, z = quant.quantize_groups(x[None], np.float32(0.75))
    # clipped range [-0.75, 0.75] -> s = 0.5, z = -0.75
    assert float(z[0]) == -0.75 and float(s[0]) == 0.5
    assert list(c[0, :4]) == [0, 3, 2, 2]          # 0.25 -> t = 2; 0 -> t = 1.5 -> 2


def test_constant_group_gives_zero_scale():
    x = np.full(128, 0.3, dtype=np.float32)
    c, s, z = quant.quantize_groups(x[None], np.float32(1.0))
    assert float(s[0]) == 0.0 and np.all(c == 0)
    assert float(z[0]) == float(np.float16(0.3))


def test_signed_zero_is_canonical():
    x = np.zeros(128, dtype=np.float32)
    x[:64] = -0.0
    c, s, z = quant.quantize_groups(x[None], np.float32(1.0))
    assert z.view(np.uint16)[0] == 0 and s.view(np.uint16)[0] == 0


def test_fp16_round_to_nearest_even():
    # 1 + 2^-11 is halfway between 1 and 1 + 2^-10: ties go to the even mantissa
    assert float(np.float32(1 + 2 ** -11).astype(np.float16)) == 1.0
    assert float(np.float32(1 + 3 * 2 ** -11).astype(np.float16)) == 1 + 2 ** -9
    assert float(np.float32(1 + 2 ** -11 + 2 ** -20).astype(np.float16)) == 1 + 2 ** -10


def test_nearest_level_brute_force():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal((400, 128)) * rng.uniform(0.1, 10, (400, 1))).astype(np.float32)
    tau = np.float32(6.0)
    c, s, z = quant.quantize_groups(x, tau)
    t = quant.t_values(x, tau, s, z)
    xc = np.clip(x.astype(np.float64), -6.0, 6.0)
    levels = z.astype(np.float64)[:, None, None] + s.astype(np.float64)[:, None, None] * np.arange(4)[None, None, :]
    dist = np.abs(xc[:, :, None] - levels)
    best = dist.argmin(axis=-1)
    near_tie = np.abs(t - np.round(t - 0.5) - 0.5) < 1e-5
    mism = (best != c) & ~near_tie
    assert not mism.any()
    # reconstruction error bound inside the representable range
    xh = quant.dequantize(c, s, z)
    inside = (xc >= z.astype(np.float64)[:, None]) & (xc <= (z.astype(np.float64) + 3 * s.astype(np.float64))[:, None])
    err = np.abs(xh - xc)
    bound = np.broadcast_to(s.astype(np.float64)[:, None] * 0.5000001, err.shape)
    assert inside.mean() > 0.9
    assert np.all(err[inside] <= bound[inside])


def test_reconstruction_bound_outside_range():
    # values below z (fp16 rounding of the minimum upwards) or above z + 3 s
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((300, 128)) * 3).astype(np.float32)
    c, s, z = quant.quantize_groups(x, np.float32(4.0))
    xc = np.clip(x.astype(np.float64), -4, 4)
    xh = quant.dequantize(c, s, z)
    mn = xc.min(1)
    mx = xc.max(1)
    slack = np.abs(z.astype(np.float64) - mn) + np.abs(3 * s.astype(np.float64) - (mx - mn))
    assert np.all(np.abs(xh - xc) <= s.astype(np.float64)[:, None] / 2 + slack[:, None] + 1e-12)


def test_rotate_to_fp32_matches_exact_rationals():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((3, 128)).astype(np.float32).astype(np.float64)
    x = x.astype(np.float32).view(np.uint32)
    x = ((x >> 16) << 16).view(np.float32).astype(np.float64)          # bf16 values
    r = rng.standard_normal((128, 128)).astype(np.float32).astype(np.float64) / 11
    got = quant.rotate_to_fp32(x, r)
    for i in range(3):
        for j in range(0, 128, 7):
            exact = sum(Fraction(float(x[i, t])) * Fraction(float(r[t, j])) for t in range(128))
            assert got[i, j] == quant._round_fraction_to_fp32(exact)


def test_rotate_to_fp32_exact_midpoint_case():
    # exact value 1 + 2^-24 is an fp32 midpoint: ties to even -> 1.0; 1 + 3*2^-24 -> 1 + 2^-22
    x = np.zeros((2, 128))
    x[:, 0] = 1.0
    x[:, 1] = 1.0
    r = np.zeros((128, 128))
    r[0, 0] = 1.0
    r[1, 0] = 2.0 ** -24
    r[0, 1] = 1.0
    r[1, 1] = 3 * 2.0 ** -24
    y = quant.rotate_to_fp32(x, r)
    assert y[0, 0] == np.float32(1.0)
    assert y[0, 1] == np.float32(1 + 2 ** -22)


def test_rotation_by_identity_is_exact():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((5, 128)).astype(np.float32).astype(np.float64)
    assert np.array_equal(quant.rotate_to_fp32(x, np.eye(128)), x.astype(np.float32))


def test_meta_bytes_roundtrip():
    s = np.array([1.0, 0.5, 65504.0], dtype=np.float16)
    z = np.array([-1.5, 2.0 ** -24, -0.0], dtype=np.float16)
    m = layout.meta_bytes(s, z)
    assert list(m[0]) == [0x00, 0x3C, 0x00, 0xBE]                     # 1.0 = 0x3C00, -1.5 = 0xBE00
    s2, z2 = layout.meta_to_sz(m)
    assert np.array_equal(s2.view(np.uint16), s.view(np.uint16)) and np.array_equal(z2.view(np.uint16), z.view(np.uint16))


@pytest.mark.parametrize("plant", ["bit_order", "truncate"])
def test_planted_quantiser_mistakes_are_caught(plant, monkeypatch):
    if plant == "bit_order":
        def bad_pack(codes):
            c = codes.astype(np.uint32).reshape(codes.shape[:-1] + (32, 4))
            b = np.zeros(c.shape[:-1], dtype=np.uint32)
            for i in range(4):
                b |= c[..., i] << (6 - 2 * i)
            return b.astype(np.uint8)
        monkeypatch.setattr(layout, "pack_codes", bad_pack)
        with pytest.raises(AssertionError):
            test_closed_form_four_levels_and_byte_order()
    else:
        monkeypatch.setattr(quant.np, "rint", np.floor)
        with pytest.raises(AssertionError):
            test_round_half_to_even_ties()
