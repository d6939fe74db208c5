"""Failure detection on the GPU without a fault.

Both cases make the failure in data the host controls and check that the
kernels turn it into a status the host reads, with the device still usable:

  * a page copy that is never issued (the decode's failure-detection hook) with
    a short wait limit: the bounded wait runs out, the launch reports
    OSCAR_ERR_TIMEOUT, and the next launch (hooks back at their defaults) gives
    exactly the output of a clean launch;
  * an out-of-range page id written into the device page table: the decode's
    own bounds check reports OSCAR_ERR_DEVICE_CHECK and skips that page (a copy of
    page 0 keeps the ring's sequence), so the output stays finite; with the id
    restored the next launch is exact again.

No test here traps, asserts on the device or touches an invalid address.
"""
import numpy as np
import pytest

from tests import parity

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def b():
    from bit_rotated_kv_decode_gb300 import binding, build
    build.build()
    binding.load()
    return binding


def _setup(b, lengths, hq=32, group=128):
    from tests.test_gpu_parity import Setup
    s = Setup(b, hq=hq, hkv=8, max_req=len(lengths), max_pages=512, pages=512 * len(lengths), seed=0x5EED,
              group=group)
    reqs = [s.open() for _ in lengths]
    for r, t in zip(reqs, lengths):
        s.prefill(r, 0, t)
    return s, reqs


def _decode(s, reqs, q):
    out = torch.full((len(reqs), s.hq, 128), float("nan"), dtype=torch.float32, device="cuda")
    s.cache.decode(0, reqs, q, out, s.b.new_workspace(s.cache.workspace_bytes(reqs)))
    return out


@pytest.mark.parametrize("hold", [0, 1])
def test_held_copy_times_out_then_next_launch_is_clean(b, hold):
    from bit_rotated_kv_decode_gb300 import synth
    # 20000 tokens x 8 kv heads: about 19 cost units per CTA on the history pages,
    # so warp 0 of most such CTAs has one or two page copies (hold 0: the first,
    # with the second in flight where there is one; hold 1: the second, after the
    # first was consumed)
    s, reqs = _setup(b, [20000])
    q = synth.queries(0, 0, s.hq, len(reqs), 0, device="cuda")
    clean = _decode(s, reqs, q)
    s.cache.check()
    clean = clean.cpu().numpy()

    s.cache.debug_decode_hooks(wait_limit=64, hold_copy=hold)
    _decode(s, reqs, q)
    with pytest.raises(b.OscarError) as e:
        s.cache.check()
    assert e.value.status == b.OSCAR_ERR_TIMEOUT
    assert "wait timed out" in str(e.value)

    # defaults back: the error word was cleared by the check, the barriers are set
    # up afresh by the next launch, and its output is bit-identical to the clean one
    s.cache.debug_decode_hooks()
    again = _decode(s, reqs, q)
    s.cache.check()
    again = again.cpu().numpy()
    assert np.array_equal(again, clean)
    parity.check_output(again[0], s.oracle_decode(reqs[0], 0, q[0]))


def test_hook_values_are_checked(b):
    s, _ = _setup(b, [100])
    for wl, hold in ((0, -1), (10, -2), ((1 << 24) + 1, -1)):
        with pytest.raises(b.OscarError) as e:
            s.cache.debug_decode_hooks(wait_limit=wl, hold_copy=hold)
        assert e.value.status == b.OSCAR_ERR_INVALID_ARG


@pytest.mark.parametrize("bad", ["past_end", "negative"])
@pytest.mark.parametrize("group", [128, 64])
def test_bad_page_id_is_reported_and_output_stays_finite(b, bad, group):
    from bit_rotated_kv_decode_gb300 import synth
    s, reqs = _setup(b, [3000, 1500], group=group)
    q = synth.queries(0, 0, s.hq, len(reqs), 0, device="cuda")
    clean = _decode(s, reqs, q)
    s.cache.check()
    clean = clean.cpu().numpy()

    pt = s.cache.device_page_table()
    r = reqs[0]
    saved = int(pt[r, 1].item())
    pt[r, 1] = s.cache.cfg.num_int2_pages + 7 if bad == "past_end" else -3
    torch.cuda.synchronize()
    out = _decode(s, reqs, q)
    with pytest.raises(b.OscarError) as e:
        s.cache.check()
    assert e.value.status == b.OSCAR_ERR_DEVICE_CHECK
    assert "error bits 0x1 " in str(e.value)
    got = out.cpu().numpy()
    assert np.isfinite(got).all()
    # the other request never read the bad entry
    assert np.array_equal(got[1], clean[1])

    pt[r, 1] = saved
    torch.cuda.synchronize()
    again = _decode(s, reqs, q)
    s.cache.check()
    assert np.array_equal(again.cpu().numpy(), clean)
    s.check_pages(r, 0)
