"""Prefill-quantize on inputs built to stress the rotation's error bound.

The prefill rotation runs on the tensor cores (bf16 products, fp32 accumulation
with a per-step truncation model) and takes its decisions from intervals around
the computed value.  These inputs spread the exponents of k across 2^-10 .. 2^2
within a token, add outlier channels and mix in exactly representable small
integers (many products cancel), so the accumulation's alignment and
truncation are exercised far beyond the synthetic workloads.  The codes, scales,
zeros and page tables must still equal the oracle's bit for bit.
"""
import numpy as np
import pytest

from tests.test_gpu_parity import Setup

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def b():
    from bit_rotated_kv_decode_gb300 import binding, build
    build.build()
    binding.load()
    return binding


def adversarial_tokens(n, hkv, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    x = torch.randn(n, hkv, 128, generator=g, dtype=torch.float64)
    expo = torch.randint(-10, 3, (n, hkv, 128), generator=g).to(torch.float64)
    x = x * torch.pow(2.0, expo)
    # outlier channels and a share of tokens made of small integers (exact cancellations)
    x[:, :, 7] *= 24.0
    x[:, :, 99] *= -24.0
    ints = torch.randint(-3, 4, (n, hkv, 128), generator=g).to(torch.float64)
    mask = (torch.arange(n) % 5 == 0).view(n, 1, 1)
    x = torch.where(mask, ints, x)
    return x.to(torch.bfloat16).cuda()


def test_prefill_bit_exact_on_wide_exponent_spread(b):
    s = Setup(b, cfg_id=0, hq=32, hkv=8, max_req=1, max_pages=80, pages=160, seed=5)
    r = s.open()
    n = 64 + 64 * 64 + 256 + 37          # 64 history pages plus a ragged tail
    k = adversarial_tokens(n, 8, 11)
    v = adversarial_tokens(n, 8, 12)
    s.cache.prefill(r, 0, k, v)
    s.mirror.prefill(r, 0, n)
    s.tokens[(r, 0)] = (k, v)
    s.cache.check()
    st = s.check_pages(r, 0)
    assert st["codes"] == (n - 320) * 8 * 2 * 128
    assert st["code_exempt"] == 0 and st["meta_exempt"] == 0, st
