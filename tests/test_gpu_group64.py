"""G_K = 64 (two quantisation groups per token-head) through the GPU path.

"Together AI Open-Sources OSCAR" (MarkTechPost), section "What OSCAR Does
Differently": per-token asymmetric INT2 with G_K = 64 channels per group.  The
cache then stores two {fp16 s, fp16 z} pairs per token-head (5120-byte
records).  Codes, scales, zeros and page tables from prefill-quantize, single
appends (with their fused demotion), explicit and multi-layer demotion must
equal the oracle's per-group quantiser bit for bit.
"""
import pytest

from tests.test_gpu_parity import Setup
from tests.test_gpu_prefill_adversarial import adversarial_tokens

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def b():
    from bit_rotated_kv_decode_gb300 import binding, build
    build.build()
    binding.load()
    return binding


def _exact(st):
    assert st["code_exempt"] == 0 and st["meta_exempt"] == 0, st


def test_group64_layout(b):
    s = Setup(b, layers=1, max_req=1, pages=8, group=64)
    lay = s.cache.layout()
    assert lay.int2_record_bytes == 5120 and lay.int2_page_stride == 8 * 5120
    assert tuple(s.cache.int2_pool(0).shape) == (8, 8, 5120)


def test_group64_write_path_bit_exact(b):
    s = Setup(b, layers=2, max_req=4, pages=300, group=64)
    lengths = [64 + 256 + 64 * 3 - 2, 1500, 40, 700]
    reqs = [s.open() for _ in lengths]
    for layer in range(2):
        for r, n in zip(reqs, lengths):
            s.prefill(r, layer, n)
    for step in range(5):            # appends across a page boundary (fused demotion)
        for layer in range(2):
            s.append(reqs, layer, step)
    busy = [reqs[0], reqs[1], reqs[3]]
    s.cache.demote(0, busy)
    for r in busy:
        s.mirror.demote(r, 0)
    s.cache.demote_layers(0, 2, busy)
    for layer in range(2):
        for r in busy:
            s.mirror.demote(r, layer)
    s.cache.check()
    for layer in range(2):
        for r in reqs:
            _exact(s.check_pages(r, layer))


def test_group64_prefill_adversarial(b):
    s = Setup(b, cfg_id=0, hq=32, hkv=8, max_req=1, max_pages=80, pages=160, seed=5, group=64)
    r = s.open()
    n = 64 + 64 * 64 + 256 + 37
    k = adversarial_tokens(n, 8, 21)
    v = adversarial_tokens(n, 8, 22)
    s.cache.prefill(r, 0, k, v)
    s.mirror.prefill(r, 0, n)
    s.tokens[(r, 0)] = (k, v)
    s.cache.check()
    _exact(s.check_pages(r, 0))


@pytest.mark.parametrize("hq", [32, 64, 8, 16])
def test_group64_decode_matches_oracle(b, hq):
    # ragged lengths: sink only, sink + part of the window, one partial history page,
    # several shuffled pages with a ragged tail
    from tests import parity
    s = Setup(b, layers=2, hq=hq, hkv=8, max_req=5, max_pages=64, pages=400, seed=0xBEEF, group=64)
    lengths = [30, 320, 449, 1700, 2600]
    reqs = [s.open() for _ in lengths]
    for layer in range(2):
        for r, n in zip(reqs, lengths):
            s.prefill(r, layer, n + layer)
        s.append(reqs, layer, 0)
    for layer in range(2):
        q, out = s.decode(reqs, layer)
        for i, r in enumerate(reqs):
            parity.check_output(out[i].cpu().numpy(), s.oracle_decode(r, layer, q[i]))


def test_group64_fused_step_matches_oracle(b):
    from bit_rotated_kv_decode_gb300 import synth
    from tests import parity
    s = Setup(b, layers=1, hq=32, hkv=8, max_req=3, pages=300, group=64)
    reqs = [s.open() for _ in range(3)]
    for r, n in zip(reqs, [64 + 256 + 64 * 2 - 1, 900, 100]):
        s.prefill(r, 0, n)
    ws = b.new_workspace(s.cache.workspace_bytes(reqs) + (1 << 16))
    for step in range(3):
        k = torch.stack([s.kv(0, s.mirror.reqs[r].T[0], 1, 100 + r)[0][0] for r in reqs])
        v = torch.stack([s.kv(0, s.mirror.reqs[r].T[0], 1, 100 + r)[1][0] for r in reqs])
        q = synth.queries(0, 0, 32, len(reqs), step, device="cuda")
        out = torch.full((len(reqs), 32, 128), float("nan"), dtype=torch.float32, device="cuda")
        s.cache.step(0, reqs, k, v, q, out, ws)
        for i, r in enumerate(reqs):
            s.mirror.append(r, 0)
            ok, ov = s.tokens[(r, 0)]
            s.tokens[(r, 0)] = (torch.cat([ok, k[i:i + 1]]), torch.cat([ov, v[i:i + 1]]))
        s.cache.check()
        for i, r in enumerate(reqs):
            parity.check_output(out[i].cpu().numpy(), s.oracle_decode(r, 0, q[i]))
    for r in reqs:
        _exact(s.check_pages(r, 0))
