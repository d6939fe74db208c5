"""The fused decode step (oscar_decode_step) against append + decode_attention.

Two caches built identically; one takes separate append and decode calls, the
other the fused step.  The cache bytes must stay identical after every step
(the append part is the same code) and the outputs must agree within the
output tolerance; the fused outputs are also checked against the oracle.
"""
import numpy as np
import pytest

from bit_rotated_kv_decode_gb300 import synth
from tests import parity
from tests.test_gpu_parity import Setup

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def b():
    from bit_rotated_kv_decode_gb300 import binding, build
    build.build()
    binding.load()
    return binding


def _pair(b, lengths, hq=32, max_req=4, pages=256):
    a = Setup(b, hq=hq, max_req=max_req, pages=pages)
    f = Setup(b, hq=hq, max_req=max_req, pages=pages)
    ra, rf = [a.open() for _ in lengths], [f.open() for _ in lengths]
    assert ra == rf
    for r, t in zip(ra, lengths):
        a.prefill(r, 0, t)
        f.prefill(r, 0, t)
    return a, f, ra


def _new_token(s, reqs):
    k = torch.stack([s.kv(0, s.mirror.reqs[r].T[0], 1, 100 + r)[0][0] for r in reqs])
    v = torch.stack([s.kv(0, s.mirror.reqs[r].T[0], 1, 100 + r)[1][0] for r in reqs])
    return k, v


def _same_cache(a, f, reqs):
    """Every byte a request uses (pages are compared where written; the rest of a
    pool holds whatever the allocation left there)."""
    pa, pf = a.cache.int2_pool(0).cpu().numpy(), f.cache.int2_pool(0).cpu().numpy()
    ba, bfp = a.cache.bf16_pool(0).cpu().numpy(), f.cache.bf16_pool(0).cpu().numpy()
    for r in reqs:
        pt, bfpt = a.cache.pages(r)
        assert (pt, bfpt) == f.cache.pages(r)
        T, he = a.cache.length(r, 0)
        assert (T, he) == f.cache.length(r, 0)
        nh = he - 64
        for pi, page in enumerate(pt):
            rows = min(64, nh - 64 * pi)
            if rows <= 0:
                continue
            assert np.array_equal(parity.slot_bytes(pa[page], rows), parity.slot_bytes(pf[page], rows)), (r, pi)
        for p in list(range(min(T, 64))) + list(range(max(he, 64), T)):
            if p < 64:
                page, row = bfpt[0], p
            else:
                slot = (p - 64) % 256
                page, row = bfpt[1 + slot // 64], slot % 64
            assert np.array_equal(ba[page, :, :, row], bfp[page, :, :, row]), (r, p)


def _steps(b, a, f, reqs, n_steps, hq):
    ws = b.new_workspace(a.cache.workspace_bytes(reqs) + (1 << 16))
    ws_f = b.new_workspace(f.cache.workspace_bytes(reqs) + (1 << 16))
    for step in range(n_steps):
        k, v = _new_token(a, reqs)
        q = synth.queries(0, 0, hq, len(reqs), step, device="cuda")
        out_a = torch.full((len(reqs), hq, 128), float("nan"), dtype=torch.float32, device="cuda")
        out_f = torch.full_like(out_a, float("nan"))
        a.cache.append(0, reqs, k, v)
        a.cache.decode(0, reqs, q, out_a, ws)
        f.cache.step(0, reqs, k, v, q, out_f, ws_f)
        for s in (a, f):
            for i, r in enumerate(reqs):
                s.mirror.append(r, 0)
                ok, ov = s.tokens[(r, 0)]
                s.tokens[(r, 0)] = (torch.cat([ok, k[i:i + 1]]), torch.cat([ov, v[i:i + 1]]))
        a.cache.check()
        f.cache.check()
        _same_cache(a, f, reqs)
        parity.check_output(out_f.cpu().numpy(), out_a.cpu().numpy())
    return q, out_f


def test_step_matches_append_then_decode_across_a_page_boundary(b):
    # 64 + 256 + 3 * 64 - 2 tokens: the third demotion opens a new history page
    lengths = [64 + 256 + 3 * 64 - 2, 300, 1000]
    a, f, reqs = _pair(b, lengths)
    q, out = _steps(b, a, f, reqs, 5, 32)
    for i, r in enumerate(reqs):
        f.check_pages(r, 0)
        parity.check_output(out[i].cpu().numpy(), f.oracle_decode(r, 0, q[i]))


def test_step_gqa8(b):
    a, f, reqs = _pair(b, [700, 129], hq=64)
    q, out = _steps(b, a, f, reqs, 3, 64)
    for i, r in enumerate(reqs):
        parity.check_output(out[i].cpu().numpy(), f.oracle_decode(r, 0, q[i]))


def test_step_batch_beyond_one_launch(b):
    # 50 requests: two launches of the fused step (48 + 2)
    lengths = [330 + 7 * (i % 5) for i in range(50)]
    a, f, reqs = _pair(b, lengths, max_req=50, pages=400)
    q, out = _steps(b, a, f, reqs, 2, 32)
    for i in (0, 47, 48, 49):
        parity.check_output(out[i].cpu().numpy(), f.oracle_decode(reqs[i], 0, q[i]))


def test_step_rejects_small_workspace_without_side_effects(b):
    a, f, reqs = _pair(b, [1000])
    k, v = _new_token(f, reqs)
    q = synth.queries(0, 0, 32, 1, 0, device="cuda")
    out = torch.empty((1, 32, 128), dtype=torch.float32, device="cuda")
    before = f.cache.length(reqs[0], 0)
    with pytest.raises(b.OscarError):
        f.cache.step(0, reqs, k, v, q, out, b.new_workspace(256))
    assert f.cache.length(reqs[0], 0) == before
