"""The uncompressed BF16 paged decode baseline against exact attention.

oscar_bf16_decode attends over every cached BF16 token; the reference is the
oracle's float64 softmax attention over the same bf16 values.  Pages are shuffled, the
lengths ragged (a partial last page, a request shorter than one sub-page), and
every row past a request's length holds NaN bit patterns, which must never
reach the output.
"""
import numpy as np
import pytest

from oracle import attention
from tests import parity

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def b():
    from bit_rotated_kv_decode_gb300 import binding, build
    build.build()
    binding.load()
    return binding


def exact(q, k, v, hkv):
    hq, d = q.shape
    g = hq // hkv
    return np.stack([attention.softmax_attention(q[h], k[:, h // g], v[:, h // g], 1.0 / np.sqrt(d))
                     for h in range(hq)])


@pytest.mark.parametrize("hq,hkv", [(32, 8), (64, 8), (8, 8), (16, 8)])
def test_bf16_decode_matches_exact_attention(b, hq, hkv):
    lens = [1000, 4096 + 37, 11, 64]
    max_pages = max((t + 63) // 64 for t in lens)
    pages = sum((t + 63) // 64 for t in lens) + 5
    g = torch.Generator(device="cpu").manual_seed(hq + hkv)
    kv = torch.full((pages, hkv, 2, 64, 128), float("nan"), dtype=torch.bfloat16)
    perm = torch.randperm(pages, generator=g).tolist()
    pt = torch.full((len(lens), max_pages), -1, dtype=torch.int32)
    toks = []
    nxt = 0
    for i, t in enumerate(lens):
        k = torch.randn(t, hkv, 128, generator=g) * 1.5
        v = torch.randn(t, hkv, 128, generator=g)
        k[:, :, 5] *= 12.0
        k, v = k.to(torch.bfloat16), v.to(torch.bfloat16)
        toks.append((k, v))
        for p in range((t + 63) // 64):
            page = perm[nxt]
            nxt += 1
            pt[i, p] = page
            rows = min(64, t - 64 * p)
            kv[page, :, 0, :rows] = k[64 * p:64 * p + rows].transpose(0, 1)
            kv[page, :, 1, :rows] = v[64 * p:64 * p + rows].transpose(0, 1)
    pt[pt < 0] = 0
    q = (torch.randn(len(lens), hq, 128, generator=g) * 0.8).to(torch.bfloat16)
    out = torch.full((len(lens), hq, 128), float("nan"), dtype=torch.float32, device="cuda")
    ws = b.bf16_decode(kv.cuda(), pt.cuda(), lens, q.cuda(), out, hkv)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 0
    got = out.cpu().numpy()
    assert np.isfinite(got).all()
    for i, (k, v) in enumerate(toks):
        ref = exact(parity.bf16_to_f64(q[i]), parity.bf16_to_f64(k), parity.bf16_to_f64(v), hkv)
        parity.check_output(got[i], ref)


def test_bf16_decode_rejects_bad_arguments(b):
    kv = torch.zeros((4, 8, 2, 64, 128), dtype=torch.bfloat16, device="cuda")
    pt = torch.zeros((1, 2), dtype=torch.int32, device="cuda")
    q = torch.zeros((1, 24, 128), dtype=torch.bfloat16, device="cuda")   # 24 / 8 = 3: not supported
    out = torch.zeros((1, 24, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(b.OscarError):
        b.bf16_decode(kv, pt, [100], q, out, 8)
    q = torch.zeros((1, 32, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((1, 32, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(b.OscarError):
        b.bf16_decode(kv, pt, [200], q, out, 8)        # 200 tokens need 4 pages, the table has 2
