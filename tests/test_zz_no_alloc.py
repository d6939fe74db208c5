"""Decode through the fixed static scratch (oscar_decode_attention_noalloc).

Collected last on purpose: the scratch is one array per device, shared by
every cache, so this file also checks that it still works after the other
GPU tests have run their decodes.  It passes on its own as well.
"""
import numpy as np
import pytest

from tests import parity

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def b():
    from bit_rotated_kv_decode_gb300 import binding, build
    build.build()
    binding.load()
    return binding


def test_batch_above_the_fixed_scratch_is_rejected_before_any_work(b):
    # metadata-only cache: the size check comes before any device work.  The
    # records of one launch of 64 requests x 32 kv heads x 8 query heads per group
    # (2 per segment plus one per CTA, 8 x 528 bytes each) need about 18 MB
    layers, hkv, n = 1, 32, 64
    cfg = b.make_config(layers, 8 * hkv, hkv, n, 8, 4 * n, 0, 0.0, 0)
    tau = np.ones((layers, hkv), np.float32)
    lib = b.OscarCache(cfg, tau_k=tau, tau_v=tau, dry_run=True)
    reqs = [lib.open() for _ in range(n)]
    for r in reqs:
        lib.prefill(r, 0, None, None, n_tokens=400)     # one history page each
    with pytest.raises(b.OscarError) as e:
        lib.decode_noalloc(0, reqs, None, None)
    assert e.value.status == b.OSCAR_ERR_INVALID_ARG
    assert "fixed" in str(e.value)
    # a small batch of the same cache passes the check (dry run does no work)
    lib.decode_noalloc(0, reqs[:4], None, None)


@pytest.mark.gpu
@pytest.mark.parametrize("hq,lengths", [(32, [3000, 1200]), (64, [2500])])
def test_two_calls_in_a_row_match_the_workspace_entry(b, hq, lengths):
    from bit_rotated_kv_decode_gb300 import synth
    from tests.test_gpu_parity import Setup
    s = Setup(b, hq=hq, max_req=4)
    reqs = [s.open() for _ in lengths]
    for r, t in zip(reqs, lengths):
        s.prefill(r, 0, t)
    qs = [synth.queries(0, 0, hq, len(reqs), step, device="cuda") for step in (0, 1)]

    # existing entry, caller workspace
    ref = []
    for q in qs:
        out = torch.full((len(reqs), hq, 128), float("nan"), dtype=torch.float32, device="cuda")
        ws = b.new_workspace(s.cache.workspace_bytes(reqs))
        s.cache.decode(0, reqs, q, out, ws)
        s.cache.check()
        ref.append(out.cpu().numpy())

    # two fixed-scratch calls back to back on one stream, no synchronisation between them
    outs = [torch.full((len(reqs), hq, 128), float("nan"), dtype=torch.float32, device="cuda") for _ in qs]
    for q, out in zip(qs, outs):
        s.cache.decode_noalloc(0, reqs, q, out)
    s.cache.check()
    for out, r in zip(outs, ref):
        got = out.cpu().numpy()
        assert np.isfinite(got).all()
        parity.check_output(got, r)

    # and once more after an append changed every length
    s.append(reqs, 0, 0)
    q = qs[0]
    out_ws = torch.empty((len(reqs), hq, 128), dtype=torch.float32, device="cuda")
    s.cache.decode(0, reqs, q, out_ws, b.new_workspace(s.cache.workspace_bytes(reqs)))
    out_fx = torch.full_like(out_ws, float("nan"))
    s.cache.decode_noalloc(0, reqs, q, out_fx)
    s.cache.check()
    parity.check_output(out_fx.cpu().numpy(), out_ws.cpu().numpy())
    # the fixed-scratch result also stands against the oracle
    for i, r in enumerate(reqs):
        parity.check_output(out_fx[i].cpu().numpy(), s.oracle_decode(r, 0, q[i]))
