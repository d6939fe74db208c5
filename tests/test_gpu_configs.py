"""GPU parity at the sizes of the pages' workloads, one layer each.

  * Qwen3-8B write path: 32768-token prefill-quantize, then 4096 single-token
    appends (each demotes the oldest recent token); every history group,
    page-table entry and BF16 row is checked against the oracle.
  * Qwen3-4B batch of 32 with context lengths drawn from U{16384..65536} and a
    shared 4096-token prefix (fork); prefix pages are shared physically; one
    fused decode step; sampled requests against the oracle.
  * Qwen3-32B shape (64 query / 8 kv heads, GQA 8), batch 8 at 131072 tokens
    with per-channel drift; one decode step; sampled requests against the oracle.
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


def _exact(stats):
    assert stats["code_exempt"] == 0 and stats["meta_exempt"] == 0, stats


def test_qwen3_8b_prefill_32k_then_4096_demotions(b):
    s = Setup(b, cfg_id=1, hq=32, hkv=8, max_req=1, max_pages=600, pages=700, seed=1)
    r = s.open()
    s.prefill(r, 0, 32768)
    st = s.check_pages(r, 0)
    assert st["codes"] == (32768 - 320) * 8 * 2 * 128
    _exact(st)
    # 4096 single-token appends, each demoting the oldest recent token
    kn = synth.kv_tokens(1, 0, 8, "k", range(32768, 32768 + 4096), device="cuda", stream_id=7)
    vn = synth.kv_tokens(1, 0, 8, "v", range(32768, 32768 + 4096), device="cuda", stream_id=7)
    for i in range(4096):
        s.cache.append(0, [r], kn[i:i + 1], vn[i:i + 1])
        s.mirror.append(r, 0)
    ok, ov = s.tokens[(r, 0)]
    s.tokens[(r, 0)] = (torch.cat([ok, kn]), torch.cat([ov, vn]))
    s.cache.check()
    T, he = s.cache.length(r, 0)
    assert (T, he) == (32768 + 4096, 32768 + 4096 - 256)
    st = s.check_pages(r, 0)
    assert st["codes"] == (32768 + 4096 - 320) * 8 * 2 * 128
    _exact(st)


def test_qwen3_4b_batch32_ragged_with_shared_prefix(b):
    lengths = synth.request_lengths(3, 32, 16384, 65536)
    pages = sum((t - 320) // 64 + 2 for t in lengths) + 64
    s = Setup(b, cfg_id=3, hq=32, hkv=8, max_req=33, max_pages=1030, pages=pages, seed=3)
    parent = s.open()
    s.prefill(parent, 0, 4096 + 256)                # history covers the 4096-token prefix
    reqs = []
    for t in lengths:
        ch = s.fork(parent, 4096)
        s.prefill(ch, 0, t - 4096, stream_id=1000 + ch)
        reqs.append(ch)
    s.cache.close(parent)
    s.mirror.close(parent)
    pts = [s.cache.pages(r)[0] for r in reqs]
    assert all(pt[:63] == pts[0][:63] for pt in pts)   # one physical copy of the prefix
    s.append(reqs, 0, 0)
    q, out = s.decode(reqs, 0)
    got = out.cpu().numpy()
    assert np.isfinite(got).all()
    order = np.argsort(lengths)
    for i in (int(order[0]), int(order[-1])):
        parity.check_output(got[i], s.oracle_decode(reqs[i], 0, q[i]))
        _exact(s.check_pages(reqs[i], 0))


def test_qwen3_32b_gqa8_131k_with_drift(b):
    T = 131072
    s = Setup(b, cfg_id=4, hq=64, hkv=8, max_req=8, max_pages=2050, pages=8 * 2046 + 8, seed=4, drift=True,
              total_len=T)
    reqs = [s.open() for _ in range(8)]
    for r in reqs:
        s.prefill(r, 0, T)
    s.append(reqs, 0, 0)
    q, out = s.decode(reqs, 0)
    got = out.cpu().numpy()
    assert np.isfinite(got).all()
    for i in (0, 7):
        parity.check_output(got[i], s.oracle_decode(reqs[i], 0, q[i]))
