"""Pins of the oracle's allocator and cache state machine, and the pages' figures."""
import itertools
import json
import os

import numpy as np
import pytest

from oracle import alloc, layout
from oracle.cache import CacheMirror, StateError

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_figures.json")


def test_seeded_order_is_a_permutation_and_seed0_is_identity():
    assert alloc.seeded_order(10, 0) == list(range(10))
    for seed in (1, 2, 12345, 2 ** 63 + 7):
        o = alloc.seeded_order(1000, seed)
        assert sorted(o) == list(range(1000)) and o != list(range(1000))


def test_fisher_yates_reaches_every_permutation_uniformly():
    counts = {}
    n_seeds = 24000
    for seed in range(1, n_seeds + 1):
        counts[tuple(alloc.seeded_order(4, seed * 7919))] = counts.get(tuple(alloc.seeded_order(4, seed * 7919)), 0) + 1
    assert len(counts) == 24                      # Sattolo's variant would reach only the 6 cyclic ones
    expect = n_seeds / 24
    chi2 = sum((c - expect) ** 2 / expect for c in counts.values())
    assert chi2 < 60                              # 23 dof; p ~ 1e-4 at 55


def test_pool_lifo_reuse_and_refcounts():
    p = alloc.PagePool(5, 0)
    a = [p.alloc() for _ in range(3)]
    assert a == [0, 1, 2]
    p.share(1)
    p.release(1)
    assert p.free_count == 2
    p.release(1)
    p.release(0)
    assert p.alloc() == 0 and p.alloc() == 1 and p.alloc() == 3


def _mirror(seed=0, layers=2):
    return CacheMirror(layers, 8, 4, 64, 200, 40, seed)


def test_prefill_then_appends_equals_longer_prefill():
    for t, n in [(10, 100), (300, 50), (320, 1), (1000, 130), (64, 300)]:
        a = _mirror(9)
        ra = a.open()
        a.prefill(ra, 0, t)
        for _ in range(n):
            a.append(ra, 0)
        b = _mirror(9)
        rb = b.open()
        b.prefill(rb, 0, t + n)
        assert a.reqs[ra].hist_pt == b.reqs[rb].hist_pt
        assert a.reqs[ra].hist_end[0] == b.reqs[rb].hist_end[0] == max(64, t + n - 256)


def test_append_demotes_only_when_window_full():
    m = _mirror()
    r = m.open()
    acts = [m.append(r, 0) for _ in range(322)]
    assert all(a["demote"] is None for a in acts[:320])
    assert acts[320]["demote"] == 64 and acts[321]["demote"] == 65
    assert m.reqs[r].hist_pt == [0]


def test_explicit_demote_and_errors():
    m = _mirror()
    r = m.open()
    m.prefill(r, 0, 64)
    with pytest.raises(StateError):
        m.demote(r, 0)
    m.append(r, 0)
    assert m.demote(r, 0) == 64
    with pytest.raises(StateError):
        m.demote(r, 0)
    with pytest.raises(StateError):
        m.prefill(r, 1, 5) or m.prefill(r, 1, 5)


def test_fork_shares_prefix_pages_and_releases_them_last():
    m = CacheMirror(1, 8, 4, 64, 30, 40, 0)
    par = m.open()
    m.prefill(par, 0, 64 + 3 * 64 + 256)
    with pytest.raises(StateError):
        m.fork(par, 100)
    ch = m.fork(par, 64 + 2 * 64)
    assert m.reqs[ch].hist_pt == m.reqs[par].hist_pt[:2]
    assert m.reqs[ch].bf16_pt[0] == m.reqs[par].bf16_pt[0]
    m.prefill(ch, 0, 300)
    assert m.reqs[ch].hist_pt[:2] == m.reqs[par].hist_pt[:2]
    free_before = m.int2.free_count
    m.close(par)
    assert m.int2.free_count == free_before + 1   # only the unshared third page came back
    m.close(ch)
    assert m.int2.free_count == 30


def test_out_of_pages_is_reported_before_any_change():
    m = CacheMirror(1, 8, 2, 64, 2, 10, 0)
    r = m.open()
    with pytest.raises(MemoryError):
        m.prefill(r, 0, 64 + 3 * 64 + 256)
    assert m.reqs[r].T[0] == 0 and m.int2.free_count == 2


def test_pages_figures():
    g = json.load(open(GOLDEN))
    assert layout.SINK_TOKENS == g["sink_tokens"]["value"]
    assert layout.RECENT_TOKENS == g["recent_tokens"]["value"]
    assert layout.HEAD_DIM == g["group_size"]["value"] == g["hadamard_order"]["value"]
    assert layout.HEAD_DIM // layout.CODE_BYTES == g["codes_per_byte"]["value"]
    # 72 bytes per token-head: 2.25 bits per element in history
    assert layout.RECORD_BYTES == 64 * 72 == 4608
    assert 8 * (layout.CODE_BYTES + layout.META_BYTES) / layout.HEAD_DIM == g["baseline_int2_bpe"]["value"]
    for key in ("bpe_128k", "bpe_32k"):
        e = g[key]
        assert round(layout.bits_per_element(e["context_tokens"]), e["round_to"]) == e["value"]
    e = g["bf16_fraction_128k_percent"]
    assert round(100 * 320 / e["context_tokens"], e["round_to"]) == e["value"]
    e = g["kv_memory_reduction"]
    assert round(16 / layout.bits_per_element(e["context_tokens"]), e["round_to"]) == e["value"]


def test_group_size_64_would_not_give_the_printed_bpe():
    """The 64-channel group reading (2.5 bits + BF16) cannot produce 2.28 at 128K."""
    bf16 = 320
    t = 131072
    bpe64 = (bf16 * 16 + (t - bf16) * (2 + 32 / 64)) / t
    assert round(bpe64, 2) != 2.28
