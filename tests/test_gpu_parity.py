"""GPU parity: the CUDA write and decode paths against the float64 oracle.

All calls go through the C ABI (ctypes binding).  Inputs are drawn by the
seeded generator on the device and copied to the host for the oracle; the
rotations and thresholds come from the oracle's own calibration builder.
"""
import numpy as np
import pytest

from bit_rotated_kv_decode_gb300 import synth
from oracle import attention, layout, rotation
from oracle.cache import CacheMirror
from tests import parity

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def b():
    from bit_rotated_kv_decode_gb300 import binding, build
    build.build()
    binding.load()
    return binding


def rotations(cfg_id, layers, hq, hkv, drift=False):
    rk, rv, tk, tv = [], [], [], []
    for layer in range(layers):
        q, k, v = synth.calibration_set(cfg_id, layer, hq, hkv, 512, drift)
        a, bb, c, d = rotation.build_layer_rotations(q, k, v, 0.9, 0.9)
        rk.append(a.astype(np.float32))
        rv.append(bb.astype(np.float32))
        tk.append(c)
        tv.append(d)
    return np.stack(rk), np.stack(rv), np.stack(tk), np.stack(tv)


class Setup:
    def __init__(self, b, cfg_id=0, layers=1, hq=32, hkv=8, max_req=4, max_pages=64, pages=256, seed=0,
                 drift=False, total_len=0, group=128, rot=None):
        self.b = b
        self.group = group
        self.cfg_id, self.L, self.hq, self.hkv = cfg_id, layers, hq, hkv
        self.drift, self.total_len = drift, total_len
        # rot: (rk, rv, tk, tv) in place of the calibrated OSCAR rotations
        self.rk, self.rv, self.tk, self.tv = rot if rot is not None else rotations(cfg_id, layers, hq, hkv, drift)
        cfg = b.make_config(layers, hq, hkv, max_req, max_pages, pages, 0, 0.0, seed, group_size=group)
        self.cache = b.OscarCache(cfg, torch.from_numpy(self.rk).cuda(), torch.from_numpy(self.rv).cuda(),
                                  self.tk, self.tv)
        self.mirror = CacheMirror(layers, hkv, max_req, max_pages, pages, 5 * max_req, seed)
        self.tokens = {}   # (req, layer) -> (k, v) device bf16 [T][Hkv][128]

    def kv(self, layer, start, n, stream_id):
        k = synth.kv_tokens(self.cfg_id, layer, self.hkv, "k", range(start, start + n), total_len=self.total_len,
                            drift=self.drift, device="cuda", stream_id=stream_id)
        v = synth.kv_tokens(self.cfg_id, layer, self.hkv, "v", range(start, start + n), total_len=self.total_len,
                            drift=self.drift, device="cuda", stream_id=stream_id)
        return k, v

    def open(self):
        r = self.cache.open()
        assert self.mirror.open() == r
        for layer in range(self.L):
            self.tokens[(r, layer)] = (torch.empty(0, self.hkv, 128, dtype=torch.bfloat16, device="cuda"),) * 2
        return r

    def prefill(self, r, layer, n, stream_id=None):
        t0 = self.mirror.reqs[r].T[layer]
        k, v = self.kv(layer, t0, n, r if stream_id is None else stream_id)
        self.cache.prefill(r, layer, k, v)
        self.mirror.prefill(r, layer, n)
        ok, ov = self.tokens[(r, layer)]
        self.tokens[(r, layer)] = (torch.cat([ok, k]), torch.cat([ov, v]))

    def append(self, reqs, layer, step):
        k = torch.stack([self.kv(layer, self.mirror.reqs[r].T[layer], 1, 100 + r)[0][0] for r in reqs])
        v = torch.stack([self.kv(layer, self.mirror.reqs[r].T[layer], 1, 100 + r)[1][0] for r in reqs])
        self.cache.append(layer, reqs, k, v)
        for i, r in enumerate(reqs):
            self.mirror.append(r, layer)
            ok, ov = self.tokens[(r, layer)]
            self.tokens[(r, layer)] = (torch.cat([ok, k[i:i + 1]]), torch.cat([ov, v[i:i + 1]]))

    def fork(self, parent, prefix):
        ch = self.cache.fork(parent, prefix)
        assert self.mirror.fork(parent, prefix) == ch
        for layer in range(self.L):
            pk, pv = self.tokens[(parent, layer)]
            self.tokens[(ch, layer)] = (pk[:prefix].clone(), pv[:prefix].clone())
        return ch

    def decode(self, reqs, layer, step=0):
        q = synth.queries(self.cfg_id, layer, self.hq, len(reqs), step, device="cuda")
        out = torch.full((len(reqs), self.hq, 128), float("nan"), dtype=torch.float32, device="cuda")
        ws = self.b.new_workspace(self.cache.workspace_bytes(reqs))
        self.cache.decode(layer, reqs, q, out, ws)
        self.cache.check()
        return q, out

    def oracle_decode(self, r, layer, q_row):
        k, v = self.tokens[(r, layer)]
        he = self.mirror.reqs[r].hist_end[layer]
        return attention.decode(parity.bf16_to_f64(q_row), parity.bf16_to_f64(k), parity.bf16_to_f64(v), he,
                                self.rk[layer].astype(np.float64), self.rv[layer].astype(np.float64),
                                self.tk[layer], self.tv[layer], group=self.group)

    def check_pages(self, r, layer, pages=None):
        """Page tables exact; every history group within the parity rules; BF16 rows exact.
        pages: history page indices to check (default all)."""
        pt, bf = self.cache.pages(r)
        assert pt == self.mirror.reqs[r].hist_pt and bf == self.mirror.reqs[r].bf16_pt
        dev_pt = self.cache.device_page_table()[r, :len(pt)].cpu().tolist()
        assert dev_pt == pt
        T, he = self.cache.length(r, layer)
        assert (T, he) == (self.mirror.reqs[r].T[layer], self.mirror.reqs[r].hist_end[layer])
        k, v = self.tokens[(r, layer)]
        kf, vf = parity.bf16_to_f64(k), parity.bf16_to_f64(v)
        pool = self.cache.int2_pool(layer).cpu().numpy()
        stats = {"code_exempt": 0, "meta_exempt": 0, "codes": 0}
        nh = he - 64
        if nh > 0:
            pos = np.arange(64, he)
            if pages is not None:
                pos = pos[np.isin((pos - 64) // 64, np.asarray(pages))]
            nh = pos.size
            pages = np.array(pt)[(pos - 64) // 64]
            rows = (pos - 64) % 64
            for h in range(self.hkv):
                rec = pool[pages, h]
                fields = [layout.record_slot_fields(rec[i], int(rows[i]), self.group) for i in range(nh)]
                for which, src, rr, tau in ((0, kf, self.rk, self.tk), (1, vf, self.rv, self.tv)):
                    codes = np.stack([f[1 if which else 0] for f in fields])
                    meta = np.stack([f[3 if which else 2] for f in fields])
                    from oracle import quant
                    x32 = quant.rotate_to_fp32(src[pos, h], rr[layer, h].astype(np.float64))
                    st = parity.compare_groups(codes, meta, x32, tau[layer, h], self.group)
                    for key in stats:
                        stats[key] += st[key]
        bfp = self.cache.bf16_pool(layer).cpu()
        kb = k.view(torch.int16).cpu()
        vb = v.view(torch.int16).cpu()
        for p in list(range(min(T, 64))) + list(range(he, T) if T > 64 else []):
            if p < 64:
                page, row = bf[0], p
            else:
                slot = (p - 64) % 256
                page, row = bf[1 + slot // 64], slot % 64
            assert torch.equal(bfp[page, :, 0, row], kb[p]) and torch.equal(bfp[page, :, 1, row], vb[p]), p
        return stats


def test_two_thousand_token_single_layer(b):
    """One layer, 32/8 heads, T = 2048 (64 sink + 1728 INT2 + 256 recent), identity page order."""
    s = Setup(b)
    r = s.open()
    s.prefill(r, 0, 2048)
    stats = s.check_pages(r, 0)
    assert stats["codes"] == 1728 * 8 * 2 * 128
    q, out = s.decode([r], 0)
    ref = s.oracle_decode(r, 0, q[0])
    res = parity.check_output(out[0].cpu().numpy(), ref)
    print("parity", stats, res)


def test_prefill_equals_sequential_appends(b):
    s1 = Setup(b, max_req=1)
    s2 = Setup(b, max_req=1)
    r1 = s1.open()
    r2 = s2.open()
    k, v = s1.kv(0, 0, 700, 7)
    s1.cache.prefill(r1, 0, k, v)
    s1.mirror.prefill(r1, 0, 700)
    s1.tokens[(r1, 0)] = (k, v)
    s2.cache.prefill(r2, 0, k[:500].contiguous(), v[:500].contiguous())
    s2.mirror.prefill(r2, 0, 500)
    for p in range(500, 700):
        s2.cache.append(0, [r2], k[p:p + 1].contiguous(), v[p:p + 1].contiguous())
        s2.mirror.append(r2, 0)
    s2.tokens[(r2, 0)] = (k, v)
    assert s1.cache.length(r1, 0) == s2.cache.length(r2, 0) == (700, 444)
    a = s1.cache.int2_pool(0).cpu()
    bb = s2.cache.int2_pool(0).cpu()
    pt = s1.cache.pages(r1)[0]
    assert pt == s2.cache.pages(r2)[0]
    for i, p in enumerate(pt):
        rows = min(64, 444 - 64 - 64 * i)
        assert np.array_equal(parity.slot_bytes(a[p].numpy(), rows), parity.slot_bytes(bb[p].numpy(), rows))
    s2.check_pages(r2, 0)


@pytest.mark.parametrize("total", [1, 63, 64, 65, 320, 321, 385, 1000])
def test_decode_edge_lengths(b, total):
    s = Setup(b, max_req=1)
    r = s.open()
    s.prefill(r, 0, total)
    s.check_pages(r, 0)
    q, out = s.decode([r], 0)
    parity.check_output(out[0].cpu().numpy(), s.oracle_decode(r, 0, q[0]))


def test_appends_across_page_boundaries_and_explicit_demote(b):
    s = Setup(b, max_req=2)
    r = s.open()
    s.prefill(r, 0, 380)
    for step in range(70):
        s.append([r], 0, step)
    s.cache.demote(0, [r])
    s.mirror.demote(r, 0)
    s.cache.demote(0, [r])
    s.mirror.demote(r, 0)
    assert s.cache.length(r, 0) == (450, 450 - 254)
    s.check_pages(r, 0)
    q, out = s.decode([r], 0)
    parity.check_output(out[0].cpu().numpy(), s.oracle_decode(r, 0, q[0]))


def test_fork_shares_prefix_pages(b):
    s = Setup(b, max_req=4)
    par = s.open()
    s.prefill(par, 0, 64 + 3 * 64 + 256)
    ch = s.fork(par, 64 + 2 * 64)
    s.prefill(ch, 0, 900, stream_id=50)
    pp = s.cache.pages(par)[0]
    pc = s.cache.pages(ch)[0]
    assert pc[:2] == pp[:2] and not set(pc[2:]) & set(pp)
    for r in (par, ch):
        s.check_pages(r, 0)
    q, out = s.decode([par, ch], 0)
    for i, r in enumerate((par, ch)):
        parity.check_output(out[i].cpu().numpy(), s.oracle_decode(r, 0, q[i]))
    s.cache.close(par)
    s.mirror.close(par)
    q, out = s.decode([ch], 0, step=1)
    parity.check_output(out[0].cpu().numpy(), s.oracle_decode(ch, 0, q[0]))


@pytest.mark.parametrize("hq", [8, 16, 32, 64])
def test_ragged_batch_two_layers_shuffled_pages(b, hq):
    # every GQA group size the cache accepts (1, 2, 4, 8 query heads per kv head)
    s = Setup(b, layers=2, hq=hq, hkv=8, max_req=6, max_pages=64, pages=400, seed=0xC0FFEE)
    lengths = [30, 320, 1700, 449, 2600]
    reqs = [s.open() for _ in lengths]
    for layer in range(2):
        for r, n in zip(reqs, lengths):
            s.prefill(r, layer, n + layer)
        s.append(reqs, layer, 0)
    for layer in range(2):
        q, out = s.decode(reqs, layer)
        for i, r in enumerate(reqs):
            parity.check_output(out[i].cpu().numpy(), s.oracle_decode(r, layer, q[i]))
    s.check_pages(reqs[4], 1)


def test_device_check_is_clean_after_all_calls(b):
    s = Setup(b, max_req=1)
    r = s.open()
    s.prefill(r, 0, 500)
    s.decode([r], 0)
    s.cache.check()


def test_unwritten_rows_holding_nan_do_not_leak(b):
    """Rows outside a request's window are never written; whatever they hold (here
    NaN bit patterns in every pool byte) must not reach the output."""
    s = Setup(b, max_req=3)
    s.cache.int2_pool(0).fill_(-1)      # codes 3, fp16 scale / zero 0xffff (NaN)
    s.cache.bf16_pool(0).fill_(-1)      # bf16 0xffff (NaN)
    reqs = [s.open() for _ in range(3)]
    for r, t in zip(reqs, (40, 300, 1000)):
        s.prefill(r, 0, t)
    s.append(reqs, 0, 0)
    q, out = s.decode(reqs, 0)
    got = out.cpu().numpy()
    assert np.isfinite(got).all()
    for i, r in enumerate(reqs):
        parity.check_output(got[i], s.oracle_decode(r, 0, q[i]))
