"""Pins of the oracle's three-segment decode attention.

"Together AI Open-Sources OSCAR" (MarkTechPost), section The Serving System:
BF16 sink of 64 tokens, BF16 recent window of 256 tokens, INT2 history in
between; "TogetherAI开源OSCAR" (ModelScope), section OSCAR的设计: the BF16 and
INT2 partials are merged by an online softmax, i.e. the result is attention
over the union of the segments.
"""
import numpy as np
import pytest

from oracle import attention, rotation


def _bf16(x):
    u = np.asarray(x, dtype=np.float32).view(np.uint32)
    # round to nearest even on the upper 16 bits
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.view(np.float32).astype(np.float64)


def _problem(total, hq=4, hkv=1, seed=0):
    rng = np.random.default_rng(seed)
    k = _bf16(rng.standard_normal((total, hkv, 128)) * np.where(np.arange(128) < 4, 20, 1))
    v = _bf16(rng.standard_normal((total, hkv, 128)) * np.where(np.arange(128) % 32 == 3, 20, 1))
    q = _bf16(rng.standard_normal((hq, 128)))
    qc = rng.standard_normal((128, hq, 128))
    kc = _bf16(rng.standard_normal((128, hkv, 128)) * np.where(np.arange(128) < 4, 20, 1))
    vc = _bf16(rng.standard_normal((128, hkv, 128)) * np.where(np.arange(128) % 32 == 3, 20, 1))
    rk, rv, tk, tv = rotation.build_layer_rotations(qc, kc, vc, 0.9, 0.9)
    return q, k, v, rk.astype(np.float32).astype(np.float64), rv.astype(np.float32).astype(np.float64), rk, rv, tk, tv


def _plain(q, k, v, g):
    out = np.zeros_like(q)
    for h in range(q.shape[0]):
        out[h] = attention.softmax_attention(q[h], k[:, h // g], v[:, h // g], 1 / np.sqrt(128))
    return out


@pytest.mark.parametrize("total", [1, 63, 64, 65, 200, 320])
def test_no_int2_segment_equals_plain_attention(total):
    q, k, v, rk, rv, _, _, tk, tv = _problem(total, hq=4, hkv=2)
    hist_end = max(64, total - 256)
    assert hist_end == 64
    got = attention.decode(q, k, v, hist_end, rk, rv, tk, tv)
    assert np.abs(got - _plain(q, k, v, 2)).max() < 1e-12


def test_identity_quantiser_equals_plain_attention():
    total = 700
    q, k, v, _, _, rk64, rv64, tk, tv = _problem(total, hq=8, hkv=2, seed=1)
    got = attention.decode(q, k, v, total - 256, rk64, rv64, tk, tv, identity_quantizer=True)
    assert np.abs(got - _plain(q, k, v, 4)).max() < 1e-12


def test_int2_segment_changes_output_but_stays_close():
    total = 900
    q, k, v, rk, rv, _, _, tk, tv = _problem(total, hq=4, hkv=1, seed=2)
    got = attention.decode(q, k, v, total - 256, rk, rv, tk, tv)
    ref = _plain(q, k, v, 4)
    err = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert 1e-6 < err < 1.0


@pytest.mark.parametrize("total", [1, 64, 65, 321, 385])
def test_naive_loop_matches_vectorised(total):
    q, k, v, rk, rv, _, _, tk, tv = _problem(total, hq=2, hkv=1, seed=3)
    hist_end = max(64, total - 256)
    a = attention.decode(q, k, v, hist_end, rk, rv, tk, tv)
    b = attention.decode_naive(q, k, v, hist_end, rk, rv, tk, tv)
    assert np.abs(a - b).max() < 1e-11


def test_segment_sizes_of_the_2048_token_case():
    sink, hist, recent = attention.segments(2048, 2048 - 256)
    assert (len(sink), len(hist), len(recent)) == (64, 1728, 256)
    sink, hist, recent = attention.segments(100000, 100000 - 256)
    assert (len(sink), len(hist), len(recent)) == (64, 99680, 256)


def test_explicit_demotion_moves_tokens_between_segments():
    total = 500
    q, k, v, rk, rv, _, _, tk, tv = _problem(total, hq=4, hkv=1, seed=4)
    a = attention.decode(q, k, v, total - 256, rk, rv, tk, tv)
    b = attention.decode(q, k, v, total - 250, rk, rv, tk, tv)
    assert np.abs(a - b).max() > 0
    sink, hist, recent = attention.segments(total, total - 250)
    assert len(hist) == total - 250 - 64 and len(recent) == 250


def test_planted_gqa_index_mistake_is_caught(monkeypatch):
    q, k, v, rk, rv, _, _, tk, tv = _problem(200, hq=4, hkv=2, seed=5)
    bad = np.zeros_like(q)
    for h in range(4):
        bad[h] = attention.softmax_attention(q[h], k[:, h % 2], v[:, h % 2], 1 / np.sqrt(128))
    good = attention.decode(q, k, v, 64, rk, rv, tk, tv)
    assert np.abs(good - bad).max() > 1e-3
