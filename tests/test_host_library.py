"""Host logic of the C library (no GPU): exports, allocator, page tables, errors.

The library runs in its metadata-only mode (device_mem = NULL); page tables
and lengths must equal the oracle's allocator / state-machine mirror exactly.
"""
import os
import re

import numpy as np
import pytest

from oracle.cache import CacheMirror, StateError

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def b():
    from bit_rotated_kv_decode_gb300 import binding, build
    build.build()
    binding.load()
    return binding


def test_every_declared_symbol_is_exported(b):
    text = open(os.path.join(ROOT, "include", "oscar.h")).read()
    names = set(re.findall(r"\b(oscar_[a-z0-9_]+)\s*\(", text))
    assert len(names) >= 18
    lib = b.load()
    for name in names:
        assert hasattr(lib, name), name
    assert set(b.exported_symbols()) >= names


def _pair(b, layers=2, hkv=8, max_req=4, max_pages=64, pages=200, bf16=0, seed=0):
    cfg = b.make_config(layers, 4 * hkv, hkv, max_req, max_pages, pages, bf16, 0.0, seed)
    tau = np.ones((layers, hkv), np.float32)
    lib = b.OscarCache(cfg, tau_k=tau, tau_v=tau, dry_run=True)
    mir = CacheMirror(layers, hkv, max_req, max_pages, pages, bf16 or 5 * max_req, seed)
    return lib, mir


def _same(lib, mir, reqs, layers):
    for r in reqs:
        pt, bf = lib.pages(r)
        assert pt == mir.reqs[r].hist_pt
        assert bf == mir.reqs[r].bf16_pt
        for layer in range(layers):
            assert lib.length(r, layer) == (mir.reqs[r].T[layer], mir.reqs[r].hist_end[layer])
    assert lib.free_pages() == (mir.int2.free_count, mir.bf16.free_count)


@pytest.mark.parametrize("seed", [0, 1, 0xDEADBEEF12345])
def test_random_call_sequence_matches_mirror(b, seed):
    rng = np.random.default_rng(seed & 0xFFFF)
    lib, mir = _pair(b, layers=2, max_req=4, max_pages=40, pages=120, seed=seed)
    live = []
    for step in range(400):
        op = rng.integers(0, 11)
        try:
            if op == 0 and len(live) < 4:
                r1 = mir.open()
                r2 = lib.open()
                assert r1 == r2
                live.append(r1)
            elif op == 1 and live:
                r = live.pop(int(rng.integers(len(live))))
                mir.close(r)
                lib.close(r)
            elif op in (2, 3) and live:
                r = live[int(rng.integers(len(live)))]
                layer = int(rng.integers(2))
                n = int(rng.integers(1, 700))
                try:
                    mir.prefill(r, layer, n)
                except (StateError, MemoryError):
                    with pytest.raises(b.OscarError):
                        lib.prefill(r, layer, None, None, n_tokens=n)
                    continue
                lib.prefill(r, layer, None, None, n_tokens=n)
            elif op in (4, 5, 6, 7) and live:
                layer = int(rng.integers(2))
                batch = list(rng.choice(live, size=int(rng.integers(1, len(live) + 1)), replace=False))
                snapshot = [(mir.reqs[r].T[layer], mir.reqs[r].hist_end[layer], list(mir.reqs[r].hist_pt))
                            for r in batch]
                free0 = (mir.int2.stack[:], list(mir.int2.refs))
                try:
                    for r in batch:
                        mir.append(int(r), layer)
                except (StateError, MemoryError):
                    for r, (t, he, pt) in zip(batch, snapshot):
                        mir.reqs[r].T[layer], mir.reqs[r].hist_end[layer], mir.reqs[r].hist_pt = t, he, pt
                    mir.int2.stack, mir.int2.refs = free0
                    # the fused decode step makes exactly the append's state changes
                    call = (lambda: lib.step(layer, batch, None, None, None, None, None)) if op == 7 else \
                        (lambda: lib.append(layer, batch, None, None))
                    with pytest.raises(b.OscarError):
                        call()
                    continue
                if op == 7:
                    lib.step(layer, batch, None, None, None, None, None)
                else:
                    lib.append(layer, batch, None, None)
            elif op == 8 and live:
                r = live[int(rng.integers(len(live)))]
                layer = int(rng.integers(2))
                try:
                    mir.demote(r, layer)
                except (StateError, MemoryError):
                    with pytest.raises(b.OscarError):
                        lib.demote(layer, [r])
                    continue
                lib.demote(layer, [r])
            elif op == 10 and live:
                # multi-layer demote: both layers of a batch, all checks before any change
                batch = [int(r) for r in rng.choice(live, size=int(rng.integers(1, len(live) + 1)), replace=False)]
                snapshot = {r: ([list(mir.reqs[r].T), list(mir.reqs[r].hist_end)], list(mir.reqs[r].hist_pt))
                            for r in batch}
                free0 = (mir.int2.stack[:], list(mir.int2.refs))
                try:
                    for layer in range(2):
                        for r in batch:
                            mir.demote(r, layer)
                except (StateError, MemoryError):
                    for r, ((t, he), pt) in snapshot.items():
                        mir.reqs[r].T, mir.reqs[r].hist_end, mir.reqs[r].hist_pt = t, he, pt
                    mir.int2.stack, mir.int2.refs = free0
                    with pytest.raises(b.OscarError):
                        lib.demote_layers(0, 2, batch)
                    continue
                lib.demote_layers(0, 2, batch)
            elif op == 9 and live and len(live) < 4:
                par = live[int(rng.integers(len(live)))]
                prefix = 64 + 64 * int(rng.integers(0, 4))
                try:
                    ch = mir.fork(par, prefix)
                except (StateError, MemoryError):
                    with pytest.raises(b.OscarError):
                        lib.fork(par, prefix)
                    continue
                assert lib.fork(par, prefix) == ch
                live.append(ch)
        except MemoryError:
            continue
        _same(lib, mir, live, 2)


def test_seeded_page_order(b):
    lib, mir = _pair(b, layers=1, max_req=1, max_pages=40, pages=50, seed=12345)
    r = lib.open()
    mir.open()
    lib.prefill(r, 0, None, None, n_tokens=64 + 30 * 64 + 256)
    mir.prefill(r, 0, 64 + 30 * 64 + 256)
    pt, _ = lib.pages(r)
    assert pt == mir.reqs[r].hist_pt and pt != list(range(30)) and len(set(pt)) == 30


def test_invalid_configs_rejected(b):
    import ctypes
    lib = b.load()
    good = b.make_config(1, 32, 8, 1, 4, 8)
    assert lib.oscar_cache_device_bytes(ctypes.byref(good)) > 0
    for field, value in [("head_dim", 64), ("sink_tokens", 32), ("recent_tokens", 128), ("page_tokens", 32),
                         ("group_size", 32), ("group_size", 96), ("num_q_heads", 24), ("num_int2_pages", 0),
                         ("max_requests", 0)]:
        cfg = b.make_config(1, 32, 8, 1, 4, 8)
        setattr(cfg, field, value)
        assert lib.oscar_cache_device_bytes(ctypes.byref(cfg)) == 0, field
    # G_K = 64 is a valid geometry: 5120-byte INT2 records instead of 4608
    g64 = b.make_config(1, 32, 8, 1, 4, 8, group_size=64)
    assert lib.oscar_cache_device_bytes(ctypes.byref(g64)) > lib.oscar_cache_device_bytes(ctypes.byref(good))


def test_bad_thresholds_rejected(b):
    cfg = b.make_config(1, 32, 8, 1, 4, 8)
    for bad in (0.0, -1.0, 70000.0, float("nan")):
        tau = np.full((1, 8), bad, np.float32)
        with pytest.raises(b.OscarError):
            b.OscarCache(cfg, tau_k=tau, tau_v=np.ones((1, 8), np.float32), dry_run=True)


def test_state_errors_leave_no_side_effect(b):
    lib, mir = _pair(b, layers=1, max_req=2, max_pages=3, pages=3)
    r = lib.open()
    with pytest.raises(b.OscarError) as e:
        lib.demote(0, [r])
    assert e.value.status == b.OSCAR_ERR_STATE
    with pytest.raises(b.OscarError) as e:
        lib.prefill(r, 0, None, None, n_tokens=64 + 4 * 64 + 256)       # needs 4 pages > max 3
    assert e.value.status == b.OSCAR_ERR_INVALID_ARG
    assert lib.length(r, 0) == (0, 64) and lib.free_pages()[0] == 3
    with pytest.raises(b.OscarError):
        lib.append(0, [r, r], None, None)                               # duplicate ids
    with pytest.raises(b.OscarError):
        lib.append(0, [3], None, None)                                  # bad id
    r2 = lib.open()
    with pytest.raises(b.OscarError) as e:
        lib.open()
    assert e.value.status == b.OSCAR_ERR_OUT_OF_PAGES
    lib.prefill(r, 0, None, None, n_tokens=64 + 2 * 64 + 256)
    with pytest.raises(b.OscarError) as e:
        lib.prefill(r2, 0, None, None, n_tokens=64 + 2 * 64 + 256)     # 2 pages needed, 1 free
    assert e.value.status == b.OSCAR_ERR_OUT_OF_PAGES
    assert lib.length(r2, 0) == (0, 64)
    with pytest.raises(b.OscarError):
        lib.fork(r, 100)
    with pytest.raises(b.OscarError) as e:
        lib.fork(r, 64 + 3 * 64)                                        # beyond what the parent demoted
    assert e.value.status == b.OSCAR_ERR_STATE


def test_workspace_query(b):
    lib, _ = _pair(b, layers=2, max_req=2, max_pages=64, pages=200)
    r = lib.open()
    lib.prefill(r, 0, None, None, n_tokens=3000)
    lib.prefill(r, 1, None, None, n_tokens=100)
    nb = lib.workspace_bytes([r])
    assert nb > 256 and nb % 256 == 0


def test_group64_geometry_and_state_machine(b):
    # G_K = 64 changes the record (5120 bytes: two {s, z} per token-head) and nothing
    # in the page tables or lengths: the same calls give the same state as group 128
    from oracle import layout
    tau = np.ones((2, 8), np.float32)
    caches = []
    for group in (128, 64):
        cfg = b.make_config(2, 32, 8, 2, 64, 200, 0, 0.0, 7, group_size=group)
        caches.append(b.OscarCache(cfg, tau_k=tau, tau_v=tau, dry_run=True))
    l128, l64 = (c.layout() for c in caches)
    assert l128.int2_record_bytes == layout.record_layout(128)["record"] == 4608
    assert l64.int2_record_bytes == layout.record_layout(64)["record"] == 5120
    assert l64.int2_page_stride == 8 * 5120 and l64.int2_layer_stride >= 200 * 8 * 5120
    assert l64.total_bytes > l128.total_bytes
    for c in caches:
        r = c.open()
        c.prefill(r, 0, None, None, n_tokens=3000)
        c.prefill(r, 1, None, None, n_tokens=700)
        c.demote_layers(0, 2, [r])
        c.demote(1, [r])
    a, g = caches
    assert a.pages(0) == g.pages(0)
    assert [a.length(0, layer) for layer in range(2)] == [g.length(0, layer) for layer in range(2)]


def _bf16_plan_blocks(lens, hkv, sms):
    """Chunk plan of the BF16 baseline: the ppc (one of ceil(max pages / c)) with the
    fewest rounds of resident blocks times (ppc + 1); 3 blocks per SM."""
    nps = [(t + 63) // 64 for t in lens]
    mx, slots = max(nps), 3 * sms
    best = None
    for c in range(1, min(mx, 256) + 1):
        ppc = -(-mx // c)
        blocks = sum(hkv * max(1, -(-n // ppc)) for n in nps)
        cost = -(-blocks // slots) * (ppc + 1)
        if best is None or cost < best[0]:
            best = (cost, blocks)
    return best[1]


def test_bf16_baseline_workspace_plan(b):
    import ctypes
    import torch
    lib = b.load()
    sms = torch.cuda.get_device_properties(0).multi_processor_count if torch.cuda.is_available() else 152

    def ws(lens, hq, hkv):
        arr = (ctypes.c_int32 * len(lens))(*lens)
        return lib.oscar_bf16_decode_workspace_bytes(len(lens), arr, hq, hkv)

    for lens, hq, hkv in [([100000], 32, 8), ([40000] * 32, 32, 8), ([131072] * 8, 64, 8), ([1, 64, 65, 5000], 8, 8)]:
        g = hq // hkv
        assert ws(lens, hq, hkv) == 256 + _bf16_plan_blocks(lens, hkv, sms) * g * 132 * 4, (lens[:2], hq)
    # one wave of equal chunks at 100K on 152 SMs: 56 chunks of 28 pages per kv head
    if sms == 152:
        assert _bf16_plan_blocks([100000], 8, 152) == 448
    assert ws([], 32, 8) == 0
    assert ws([0], 32, 8) == 0
    assert ws([100], 20, 8) == 0                       # query heads not a multiple of kv heads
    assert ws([100] * 65, 32, 8) == 0                  # more than 64 requests per launch


def test_decode_hook_values_checked_on_the_host(b):
    cfg = b.make_config(1, 32, 8, 1, 4, 8)
    tau = np.ones((1, 8), np.float32)
    cache = b.OscarCache(cfg, tau_k=tau, tau_v=tau, dry_run=True)
    cache.debug_decode_hooks(wait_limit=1, hold_copy=-1)
    cache.debug_decode_hooks(wait_limit=1 << 24, hold_copy=3)
    for wl, hold in ((0, -1), ((1 << 24) + 1, -1), (100, -2)):
        with pytest.raises(b.OscarError) as e:
            cache.debug_decode_hooks(wait_limit=wl, hold_copy=hold)
        assert e.value.status == b.OSCAR_ERR_INVALID_ARG
    cache.debug_decode_hooks()
