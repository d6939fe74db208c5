"""Multi-layer demote (oscar_demote_layers) against per-layer oscar_demote.

Two caches built identically over three layers.  One demotes layer by layer,
the other demotes all layers in one call; every byte either request uses must
agree, and the history groups must match the oracle.  Then a few decode steps
in the order a model runs them: all layers' demotion at the start of the step,
then per layer the fused append + decode (which then only writes the new
token), each checked against the oracle's decode.
"""
import numpy as np
import pytest

from bit_rotated_kv_decode_gb300 import synth
from tests import parity
from tests.test_gpu_parity import Setup

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

LAYERS = 3


@pytest.fixture(scope="module")
def b():
    from bit_rotated_kv_decode_gb300 import binding, build
    build.build()
    binding.load()
    return binding


def _same_layer(a, f, reqs, layer):
    pa, pf = a.cache.int2_pool(layer).cpu().numpy(), f.cache.int2_pool(layer).cpu().numpy()
    for r in reqs:
        pt, _ = a.cache.pages(r)
        assert (pt, _) == f.cache.pages(r)
        T, he = a.cache.length(r, layer)
        assert (T, he) == f.cache.length(r, layer)
        nh = he - 64
        for pi, page in enumerate(pt):
            rows = min(64, nh - 64 * pi)
            if rows <= 0:
                continue
            assert np.array_equal(parity.slot_bytes(pa[page], rows), parity.slot_bytes(pf[page], rows)), \
                (r, layer, pi)


def _build(b, lengths):
    s = Setup(b, layers=LAYERS, max_req=4, pages=300)
    reqs = [s.open() for _ in lengths]
    for r, t in zip(reqs, lengths):
        for layer in range(LAYERS):
            s.prefill(r, layer, t)
    return s, reqs


def test_demote_layers_equals_per_layer_demote(b):
    # 64 + 256 + 64 * 3 tokens: three full history pages, so the first demotion opens a new one
    lengths = [64 + 256 + 64 * 3, 700, 333]
    a, reqs = _build(b, lengths)
    f, reqs_f = _build(b, lengths)
    assert reqs == reqs_f
    for _ in range(3):
        for layer in range(LAYERS):
            a.cache.demote(layer, reqs)
            for r in reqs:
                a.mirror.demote(r, layer)
        f.cache.demote_layers(0, LAYERS, reqs)
        for layer in range(LAYERS):
            for r in reqs:
                f.mirror.demote(r, layer)
    a.cache.check()
    f.cache.check()
    for layer in range(LAYERS):
        _same_layer(a, f, reqs, layer)
        for r in reqs:
            st = f.check_pages(r, layer)
            assert st["code_exempt"] == 0 and st["meta_exempt"] == 0, st


def test_demote_all_layers_then_fused_steps(b):
    s, reqs = _build(b, [64 + 256 + 64 * 2 - 1, 900])
    ws = b.new_workspace(s.cache.workspace_bytes(reqs) + (1 << 16))
    hq = s.hq
    for step in range(4):
        s.cache.demote_layers(0, LAYERS, reqs)
        for layer in range(LAYERS):
            for r in reqs:
                s.mirror.demote(r, layer)
        for layer in range(LAYERS):
            k = torch.stack([s.kv(layer, s.mirror.reqs[r].T[layer], 1, 100 + r)[0][0] for r in reqs])
            v = torch.stack([s.kv(layer, s.mirror.reqs[r].T[layer], 1, 100 + r)[1][0] for r in reqs])
            q = synth.queries(0, layer, hq, len(reqs), step, device="cuda")
            out = torch.full((len(reqs), hq, 128), float("nan"), dtype=torch.float32, device="cuda")
            s.cache.step(layer, reqs, k, v, q, out, ws)
            for i, r in enumerate(reqs):
                s.mirror.append(r, layer)
                ok, ov = s.tokens[(r, layer)]
                s.tokens[(r, layer)] = (torch.cat([ok, k[i:i + 1]]), torch.cat([ov, v[i:i + 1]]))
            s.cache.check()
            for i, r in enumerate(reqs):
                T, he = s.cache.length(r, layer)
                assert T - he == 256          # the window refilled by the append, nothing demoted by it
                parity.check_output(out[i].cpu().numpy(), s.oracle_decode(r, layer, q[i]))
    for layer in range(LAYERS):
        for r in reqs:
            s.check_pages(r, layer)


def test_demote_layers_errors_leave_no_change(b):
    s, reqs = _build(b, [700, 50])           # the second request is all sink: nothing to demote
    before = [s.cache.length(r, layer) for r in reqs for layer in range(LAYERS)]
    with pytest.raises(b.OscarError):
        s.cache.demote_layers(0, LAYERS, reqs)
    with pytest.raises(b.OscarError):
        s.cache.demote_layers(1, LAYERS + 1, reqs[:1])
    with pytest.raises(b.OscarError):
        s.cache.demote_layers(2, 2, reqs[:1])
    assert [s.cache.length(r, layer) for r in reqs for layer in range(LAYERS)] == before
    s.cache.check()
