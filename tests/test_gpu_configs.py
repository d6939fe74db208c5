"""GPU parity at the sizes of the pages' workloads, one layer each.

  * Qwen3-8B write path: 32768-token prefill-quantize, then 4096 single-token
    appends (each demotes the oldest recent token); every history group,
    page-table entry and BF16 row is checked against the oracle.
  * Qwen3-8B at 100000 tokens on shuffled pages: one fused decode step (append
    with demotion, then decode) through oscar_decode_step; every query head
    against the oracle; the page the demotion filled and the first page checked
    byte for byte.
  * Qwen3-4B batch of 32 with context lengths drawn from U{16384..65536} and a
    shared 4096-token prefix (fork); prefix pages are shared physically; one
    fused decode step; eight requests across the length range against the oracle.
  * Qwen3-32B shape (64 query / 8 kv heads, GQA 8), batch 8 at 131072 tokens
    with per-channel drift; one decode step; sampled requests against the oracle
    and a sample of their history pages checked byte for byte.
  * The ablation rotations (identity, Hadamard with bit reversal) through the
    write path, byte-checked against the oracle at quantisation groups 128 and 64.
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


def test_qwen3_8b_100k_one_step_every_head(b):
    T = 100000
    n_pages = (T - 320) // 64 + 3
    s = Setup(b, cfg_id=2, hq=32, hkv=8, max_req=1, max_pages=n_pages + 2, pages=n_pages + 8, seed=2)
    r = s.open()
    s.prefill(r, 0, T)
    T0, he0 = s.cache.length(r, 0)
    assert T0 - he0 == 256                           # the window is full: the step demotes
    k, v = s.kv(0, T0, 1, 100 + r)
    q = synth.queries(2, 0, 32, 1, 0, device="cuda")
    out = torch.full((1, 32, 128), float("nan"), dtype=torch.float32, device="cuda")
    s.cache.step(0, [r], k, v, q, out, b.new_workspace(s.cache.workspace_bytes([r])))
    s.cache.check()
    s.mirror.append(r, 0)
    ok, ov = s.tokens[(r, 0)]
    s.tokens[(r, 0)] = (torch.cat([ok, k]), torch.cat([ov, v]))
    T1, he1 = s.cache.length(r, 0)
    assert (T1, he1) == (T0 + 1, he0 + 1)
    got = out.cpu().numpy()[0]
    assert np.isfinite(got).all()
    parity.check_output(got, s.oracle_decode(r, 0, q[0]))
    hot = (he1 - 1 - 64) // 64                       # the page the demoted token went to
    st = s.check_pages(r, 0, pages=[0, hot])
    assert st["codes"] == (64 + (he1 - 64) - 64 * hot) * 8 * 2 * 128


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
    # eight requests across the length range, the shortest and the longest included
    for i in sorted({int(order[j]) for j in np.linspace(0, len(order) - 1, 8).round().astype(int)}):
        parity.check_output(got[i], s.oracle_decode(reqs[i], 0, q[i]))
    for i in (int(order[0]), int(order[-1])):
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
    # a sample of the drifting history, byte for byte: the first and last pages and
    # a seeded selection between them (the page of the step's demotion included)
    n_hist = (s.cache.length(reqs[7], 0)[1] - 64 + 63) // 64
    rng = np.random.default_rng(4)
    sample = sorted({0, 1, n_hist - 2, n_hist - 1, *rng.choice(n_hist, 12, replace=False).tolist()})
    st = s.check_pages(reqs[7], 0, pages=sample)
    assert st["codes"] > 0


def _ablation_rotations(variant, cfg_id=0, hq=32, hkv=8):
    """The ablation's rotations for one layer, built by the oracle: R = I (naive
    INT2) or R = H_Had P_br (no query eigenbasis), thresholds the 0.9 quantile of
    the rotated calibration set."""
    from oracle import rotation
    d = 128
    r = np.eye(d) if variant == "identity" else rotation.compose_rotation(np.eye(d), use_bit_reversal=True)
    r32 = r.astype(np.float32)
    _, kc, vc = synth.calibration_set(cfg_id, 0, hq, hkv, 512, False)
    tk = np.zeros((1, hkv), np.float32)
    tv = np.zeros((1, hkv), np.float32)
    for h in range(hkv):
        tk[0, h] = rotation.clip_threshold((kc[:, h].astype(np.float32) @ r32).astype(np.float64), 0.9)
        tv[0, h] = rotation.clip_threshold((vc[:, h].astype(np.float32) @ r32).astype(np.float64), 0.9)
    rr = np.broadcast_to(r32, (1, hkv, d, d)).copy()
    return rr, rr.copy(), tk, tv


@pytest.mark.parametrize("group", [128, 64])
@pytest.mark.parametrize("variant", ["identity", "hadamard"])
def test_ablation_rotations_write_path_byte_exact(b, variant, group):
    s = Setup(b, hq=32, hkv=8, max_req=1, max_pages=40, pages=48, seed=11, group=group,
              rot=_ablation_rotations(variant))
    r = s.open()
    s.prefill(r, 0, 2048 + 320)
    s.append([r], 0, 0)                              # one demotion through the append path too
    st = s.check_pages(r, 0)
    assert st["codes"] == (2048 + 1) * 8 * 2 * 128
