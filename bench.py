"""Benchmark of the three-segment INT2 KV-cache hot path on GB300.

Default workload (N = 1): Qwen3-8B attention shape, 32 layers, 32 query / 8 KV
heads, head_dim 128, batch 1, 100,000-token context (64 BF16 sink + 99,680
INT2 history + 256 BF16 recent), 64-token pages in a seeded random physical
order.  One step = for every layer: append one token (demoting the oldest
recent token into INT2 history) and run decode attention over the whole
cache.  Inputs are synthetic (seeded generator), resident in HBM before the
timed region; the step's data (1.9 GB) is far larger than the 129 MB L2.

Prints one JSON line.  ``--impl reference`` times the float64 oracle on the
host cores instead (a bounded sample of the same workload).
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attention µs/step & KV HBM GB/s (frac of 8 TB/s) at 100K ctx; demote tok/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
INT2_BYTES_PER_TOKEN_HEAD = 72          # 2 x (32 code bytes + 4 meta bytes)


def int2_bytes_per_token_head(group: int = 128) -> int:
    """K and V codes (2 x 32 bytes) plus one fp16 {s, z} per group of each."""
    return 2 * (32 + 4 * (128 // group))
BF16_BYTES_PER_TOKEN_HEAD = 512         # K and V rows of 128 bf16

WORKLOADS = {
    1: dict(name="qwen3-8b-32k-prefill-and-demote", layers=32, q_heads=32, kv_heads=8, batch=1, context=32768,
            write_path=True),
    2: dict(name="qwen3-8b-100k-decode", layers=32, q_heads=32, kv_heads=8, batch=1, context=100000),
    3: dict(name="qwen3-4b-b32-16k-64k-shared-4k-prefix-decode", layers=36, q_heads=32, kv_heads=8, batch=32,
            context=(16384, 65536), prefix=4096),
    4: dict(name="qwen3-32b-128k-b8-decode", layers=64, q_heads=64, kv_heads=8, batch=8, context=131072),
}


# ----------------------------------------------------------------------------------------------
def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, world: int) -> float:
    """Max of a float over all ranks (identity on one rank)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def measured_peak_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def measured_peak_bf16():
    """Dense bf16 tensor peak for a kernel timed alone (burst), TFLOP/s."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def committed_traffic(kernel: str):
    """Per-launch DRAM bytes of a kernel from the committed ncu summary, if current."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            entry = json.load(f)[kernel]
    except Exception:
        return None
    import hashlib
    h = hashlib.sha256()
    try:
        # the kernel's file and the headers it includes, in the listed order
        for name in entry["sources"] if "sources" in entry else [entry["source"]]:
            h.update(open(os.path.join(ROOT, "bit_rotated_kv_decode_gb300", "csrc", name), "rb").read())
    except OSError:
        return None
    return entry["bytes_per_launch"] if h.hexdigest()[:16] == entry.get("source_sha256_16") else None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        # raw samples: a per-process scratch file (or OSCAR_CLOCKS_CSV to keep them)
        import tempfile
        self.path = os.environ.get("OSCAR_CLOCKS_CSV") or os.path.join(
            tempfile.gettempdir(), f"oscar_clocks_rank{gpu_index}_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return None
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------------------------
def pages_for(hist_end: int) -> int:
    return (hist_end - 64 + 63) // 64 if hist_end > 64 else 0


def algorithmic_bytes(tokens: int, hist_end: int, kv_heads: int, group: int = 128) -> int:
    """Bytes one decode of one request must read: INT2 codes + fp16 meta + BF16 segments."""
    n_hist = max(0, hist_end - 64)
    n_bf16 = min(tokens, 64) + (tokens - hist_end if tokens > 64 else 0)
    return kv_heads * (n_hist * int2_bytes_per_token_head(group) + n_bf16 * BF16_BYTES_PER_TOKEN_HEAD)


class Workload:
    """The cache, its rotations and every input of the timed steps, resident on the GPU."""

    def __init__(self, cfg_id: int, steps_total: int, log, layers: int = 0, override=None, reserve: int = 0):
        import torch
        from bit_rotated_kv_decode_gb300 import binding, build, calibrate, synth
        build.build()
        self.torch = torch
        self.b = binding
        self.synth = synth
        w = dict(WORKLOADS[cfg_id], **(override or {}))
        self.cfg_id = cfg_id
        self.w = w
        self.L, self.hq, self.hkv, self.batch = w["layers"], w["q_heads"], w["kv_heads"], w["batch"]
        if isinstance(w["context"], tuple):
            self.lens = synth.request_lengths(cfg_id, self.batch, *w["context"])
        else:
            self.lens = [w["context"]] * self.batch
        self.T0 = max(self.lens)
        self.prefix = w.get("prefix", 0)
        # generator stream of each request's own tokens (0 holds a shared prefix)
        self.sid = [1 + i if self.prefix else i for i in range(self.batch)]
        if layers:
            self.L = layers
        self.drift = cfg_id == 4
        t = time.time()
        fit = None if self.L <= 32 else list(range(0, self.L, 8))
        self.rk, self.rv, self.tk, self.tv = calibrate.calibrate_model(cfg_id, self.L, self.hq, self.hkv,
                                                                       drift=self.drift, layers=fit)
        log(f"calibration {time.time() - t:.1f}s")
        # reserve: extra tokens per request (steps that reuse earlier inputs) the page pool must hold
        grow = steps_total + reserve
        max_pages = pages_for(self.T0 + grow + 64) + 1
        n_pages = sum(pages_for(t + grow + 64) + 1 for t in self.lens) + 8
        seed = synth.seed_for(cfg_id, 0, 0, 99) or 1
        self.group = w.get("group", 128)
        cfg = binding.make_config(self.L, self.hq, self.hkv, self.batch + (1 if self.prefix else 0), max_pages,
                                  n_pages, 0, 0.0, seed, group_size=self.group)
        self.cache = binding.OscarCache(cfg, torch.from_numpy(self.rk).cuda(), torch.from_numpy(self.rv).cuda(),
                                        self.tk, self.tv)
        t = time.time()

        def fill(r, layer, p0, p1, sid, total):
            k = synth.kv_tokens(cfg_id, layer, self.hkv, "k", range(p0, p1), total_len=total, drift=self.drift,
                                device="cuda", stream_id=sid)
            v = synth.kv_tokens(cfg_id, layer, self.hkv, "v", range(p0, p1), total_len=total, drift=self.drift,
                                device="cuda", stream_id=sid)
            self.cache.prefill(r, layer, k, v)

        if self.prefix:
            # one parent holds the shared prefix (demoted in every layer); each request forks it
            parent = self.cache.open()
            for layer in range(self.L):
                fill(parent, layer, 0, self.prefix + 256, 0, self.prefix + 256)
            self.reqs = [self.cache.fork(parent, self.prefix) for _ in range(self.batch)]
            self.cache.close(parent)
            for layer in range(self.L):
                for i, r in enumerate(self.reqs):
                    fill(r, layer, self.prefix, self.lens[i], self.sid[i], self.lens[i])
        else:
            self.reqs = [self.cache.open() for _ in range(self.batch)]
            for layer in range(self.L):
                for i, r in enumerate(self.reqs):
                    fill(r, layer, 0, self.lens[i], self.sid[i], self.lens[i])
        torch.cuda.synchronize()
        self.cache.check()
        log(f"prefill {time.time() - t:.1f}s")
        # inputs of every step: new k / v per layer, q per layer
        n = steps_total
        self.k_new = torch.empty((n, self.L, self.batch, self.hkv, 128), dtype=torch.bfloat16, device="cuda")
        self.v_new = torch.empty_like(self.k_new)
        self.q = torch.empty((n, self.L, self.batch, self.hq, 128), dtype=torch.bfloat16, device="cuda")
        for layer in range(self.L):
            mix = synth.query_mix(cfg_id, layer, self.hq, device="cuda")
            for i in range(self.batch):
                t0 = self.lens[i]
                self.k_new[:, layer, i] = synth.kv_tokens(cfg_id, layer, self.hkv, "k", range(t0, t0 + n),
                                                          total_len=t0, drift=self.drift, device="cuda",
                                                          stream_id=self.sid[i])
                self.v_new[:, layer, i] = synth.kv_tokens(cfg_id, layer, self.hkv, "v", range(t0, t0 + n),
                                                          total_len=t0, drift=self.drift, device="cuda",
                                                          stream_id=self.sid[i])
            for s in range(n):
                self.q[s, layer] = synth.queries(cfg_id, layer, self.hq, self.batch, s, device="cuda", mix=mix)
        self.out = torch.empty((self.L, self.batch, self.hq, 128), dtype=torch.float32, device="cuda")
        ws_bytes = self.cache.workspace_bytes(self.reqs) + (1 << 20)
        self.ws = binding.new_workspace(ws_bytes)
        self.step_index = 0
        self.fused = True
        self.demote_first = False
        # raw C entry points with pre-marshalled arguments (the binding's own calls, minus re-marshalling)
        self.lib = self.cache.lib
        self.h = self.cache.h
        self.reqs_arr = (ctypes.c_int32 * self.batch)(*self.reqs)
        self.ws_ptr = self.ws.data_ptr()
        self.ws_len = self.ws.numel()

    def stream_ptr(self):
        return self.torch.cuda.current_stream().cuda_stream

    def pointers(self, s: int):
        """Device addresses of step s's inputs and outputs, per layer (computed once per step)."""
        kn, vn, q, out = self.k_new[s], self.v_new[s], self.q[s], self.out
        return [(kn[l].data_ptr(), vn[l].data_ptr(), q[l].data_ptr(), out[l].data_ptr()) for l in range(self.L)]

    def run_step(self, ptrs, stream, dec_events=None, app_events=None):
        """One step: every layer appends (with demotion) and decodes."""
        lib, h, n, ra, ws, wl = self.lib, self.h, self.batch, self.reqs_arr, self.ws_ptr, self.ws_len
        append, decode, fused = lib.oscar_append, lib.oscar_decode_attention, lib.oscar_decode_step
        if self.demote_first and lib.oscar_demote_layers(h, 0, self.L, n, ra, stream):
            raise RuntimeError(f"demote failed: {lib.oscar_last_error(h).decode()}")
        if dec_events is None:
            for layer, (kp, vp, qp, op) in enumerate(ptrs):
                if self.fused:
                    st = fused(h, layer, n, ra, kp, vp, qp, op, ws, wl, stream)
                else:
                    st = append(h, layer, n, ra, kp, vp, stream) or decode(h, layer, n, ra, qp, op, ws, wl, stream)
                if st:
                    raise RuntimeError(f"step failed: {lib.oscar_last_error(h).decode()}")
            return
        for layer, (kp, vp, qp, op) in enumerate(ptrs):
            app_events[layer][0].record()
            st = append(h, layer, n, ra, kp, vp, stream)
            app_events[layer][1].record()
            dec_events[layer][0].record()
            st |= decode(h, layer, n, ra, qp, op, ws, wl, stream)
            dec_events[layer][1].record()
            if st:
                raise RuntimeError(f"step failed: {lib.oscar_last_error(h).decode()}")

    def decode_bytes(self, layer: int, unique: bool = True) -> int:
        """Algorithmic bytes of one layer's decode; history pages of a shared prefix count once."""
        tot = 0
        for r in self.reqs:
            t, he = self.cache.length(r, layer)
            tot += algorithmic_bytes(t, he, self.hkv, self.group)
        if unique and self.prefix:
            tot -= (self.batch - 1) * (self.prefix - 64) * self.hkv * int2_bytes_per_token_head(self.group)
        return tot


def run_gpu(args, log):
    import torch
    rank, world, local = dist_info()
    torch.cuda.set_device(local)
    W, K = args.warmup, args.steps
    ew, ek = 2, max(3, K // 2)
    wl = Workload(args.config, W + 2 * K + ew + ek, log, args.layers,
                  override={"group": args.group} if args.group != 128 else None,
                  reserve=0 if args.demote_first else 2 * DEMOTE_STEP_PAIRS)
    wl.fused = not args.separate_calls
    wl.demote_first = args.demote_first
    stream = wl.stream_ptr()
    L = wl.L
    ptrs = [wl.pointers(s) for s in range(W + 2 * K)]
    # --- device-resident timing of whole steps (no per-kernel events) --------------------------
    for s in range(W):
        wl.run_step(ptrs[s], stream)
    torch.cuda.synchronize()
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    start, end = mk(), mk()
    bytes_before = np.mean([wl.decode_bytes(layer) for layer in (0, L - 1)])
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        start.record()
        for i in range(K):
            wl.run_step(ptrs[W + i], stream)
        end.record()
        torch.cuda.synchronize()
        barrier(world)
    wl.cache.check()
    total_ms = start.elapsed_time(end)
    total_ms = max_over_ranks(total_ms, world)
    us_step = 1000.0 * total_ms / K
    # --- per-kernel durations: the same steps again, CUDA events around each call -------------
    dec = [[(mk(), mk()) for _ in range(L)] for _ in range(K)]
    app = [[(mk(), mk()) for _ in range(L)] for _ in range(K)]
    bytes_per_launch = []
    torch.cuda.synchronize()
    for i in range(K):
        wl.run_step(ptrs[W + K + i], stream, dec[i], app[i])
        bytes_per_launch.append(np.mean([wl.decode_bytes(layer) for layer in (0, L - 1)]))
    torch.cuda.synchronize()
    wl.cache.check()
    dec_us = [1000.0 * a.elapsed_time(b) for row in dec for (a, b) in row]
    app_us = [1000.0 * a.elapsed_time(b) for row in app for (a, b) in row]
    dec_avg = float(np.mean(dec_us))
    app_avg = float(np.mean(app_us))
    bpl = float(np.mean(bytes_per_launch))
    kv_bytes_step = float(np.mean([bytes_before] + bytes_per_launch)) * L
    # --- end to end: each step's inputs copied in from pinned host memory and its output
    # copied back, all inside the timed region.  The copies run on streams of their own,
    # as a serving loop would overlap them: the inputs of a step while the step before
    # computes, the output of a step while the next one computes (two output buffers
    # alternate).  The input stream starts at the region's start event, and the end
    # event follows the last output copy.
    base = W + 2 * K
    kh = wl.k_new[base:].cpu().pin_memory()
    vh = wl.v_new[base:].cpu().pin_memory()
    qh = wl.q[base:].cpu().pin_memory()
    oh = torch.empty((ew + ek,) + tuple(wl.out.shape), dtype=torch.float32).pin_memory()
    outs = [wl.out, torch.empty_like(wl.out)]
    eptrs = []
    for i in range(ew + ek):
        o = outs[i % 2]
        eptrs.append([(kp, vp, qp, o[layer].data_ptr()) for layer, (kp, vp, qp, _) in enumerate(wl.pointers(base + i))])
    main = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    in_done = [torch.cuda.Event() for _ in range(ew + ek)]
    comp_done = [torch.cuda.Event() for _ in range(ew + ek)]
    out_done = [torch.cuda.Event() for _ in range(ew + ek)]
    torch.cuda.synchronize()
    for i in range(ew + ek):
        if i == ew:
            torch.cuda.synchronize()
            barrier(world)
            e0 = mk()
            e0.record(main)
            s_in.wait_event(e0)
        with torch.cuda.stream(s_in):
            wl.k_new[base + i].copy_(kh[i], non_blocking=True)
            wl.v_new[base + i].copy_(vh[i], non_blocking=True)
            wl.q[base + i].copy_(qh[i], non_blocking=True)
            in_done[i].record(s_in)
        main.wait_event(in_done[i])
        if i >= 2:
            main.wait_event(out_done[i - 2])   # the output buffer of step i - 2 has been read
        wl.run_step(eptrs[i], stream)
        comp_done[i].record(main)
        s_out.wait_event(comp_done[i])
        with torch.cuda.stream(s_out):
            oh[i].copy_(outs[i % 2], non_blocking=True)
            out_done[i].record(s_out)
    main.wait_event(out_done[ew + ek - 1])
    e1 = mk()
    e1.record(main)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    e2e_us = 1000.0 * e2e_ms / ek
    h2d = (kh[0].numel() + vh[0].numel() + qh[0].numel()) * 2
    d2h = oh[0].numel() * 4
    peak, peak_kind = measured_peak_hbm()
    # the decode kernels' time per launch, bounded from above: in fused mode the timed
    # region's step time per layer (front + stream + merge, back to back, PDL overlap
    # intact); with separate calls the event-timed decode call (which breaks the overlap)
    launch_us = us_step / L if wl.fused else dec_avg
    achieved = bpl / (launch_us * 1e-6) / 1e9
    res = {
        "us_step": us_step, "kv_bytes_step": kv_bytes_step, "dec_avg_us": dec_avg, "app_avg_us": app_avg, "bytes_per_launch": bpl,
        "achieved_gbs": achieved, "peak": peak, "peak_kind": peak_kind, "e2e_us": e2e_us, "h2d": h2d, "d2h": d2h,
        "launch_us": launch_us,
        "clocks": clk.summary(),
        # a decode step is one kernel per launch of up to 48 requests; separate calls
        # are an append kernel (48 requests) and a decode kernel (64 requests)
        "launches": K * (L * (-(-wl.batch // 48) if wl.fused else -(-wl.batch // 48) - (-wl.batch // 64)) +
                         (-(-L * wl.batch // 96) if wl.demote_first else 0)),
        "world": world, "rank": rank,
    }
    return wl, res


DEMOTE_STEP_PAIRS = 600      # step pairs of the in-step demotion cost (about 1 s at 100K x 32 layers)
DEMOTE_MIN_MS = 1000.0       # timed region of each oscar_demote_layers rate


def demote_record(wl, log):
    """Demotion throughput, two ways.

    (1) oscar_demote_layers over all layers of the workload's shape at batch 1 and
        batch 32, as tokens x layers per second.  Each request holds a sink, a full
        recent window and one history page; a chunk of 192 calls (each demotes one
        token per request in every layer) is timed with CUDA events, then the
        requests are closed and refilled outside the timed chunks; chunks repeat
        until their summed time reaches DEMOTE_MIN_MS.
    (2) The demotion's cost inside the fused step, on the workload itself: pairs of
        whole steps (oscar_decode_step in every layer), the first with a full window
        (every append demotes), the second after one oscar_demote_layers made room
        (no append demotes); CUDA events around each step and around the
        oscar_demote_layers call.  The step inputs of earlier steps are reused."""
    import torch
    b, L, hq, hkv = wl.b, wl.L, wl.hq, wl.hkv
    lib, stream = wl.lib, wl.stream_ptr()
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    rec = {}
    # (1) standalone rates
    T0, per_chunk = 320 + 64, 192
    kk = [wl.synth.kv_tokens(wl.cfg_id, l, hkv, "k", range(0, T0), device="cuda", stream_id=5) for l in range(L)]
    vv = [wl.synth.kv_tokens(wl.cfg_id, l, hkv, "v", range(0, T0), device="cuda", stream_id=5) for l in range(L)]
    rates = {}
    for n in (1, 32):
        max_pages = pages_for(T0 + 64) + 4
        cfg = b.make_config(L, hq, hkv, n, max_pages, n * max_pages + 8, 0, 0.0, 77, group_size=wl.group)
        cache = b.OscarCache(cfg, torch.from_numpy(wl.rk).cuda(), torch.from_numpy(wl.rv).cuda(), wl.tk, wl.tv)
        h = cache.h
        timed_ms, chunks = 0.0, 0
        while timed_ms < DEMOTE_MIN_MS:
            reqs = [cache.open() for _ in range(n)]
            for l in range(L):
                for r in reqs:
                    cache.prefill(r, l, kk[l], vv[l])
            ra = (ctypes.c_int32 * n)(*reqs)
            e0, e1 = mk(), mk()
            torch.cuda.synchronize()
            e0.record()
            for _ in range(per_chunk):
                if lib.oscar_demote_layers(h, 0, L, n, ra, stream):
                    raise RuntimeError(lib.oscar_last_error(h).decode())
            e1.record()
            torch.cuda.synchronize()
            cache.check()
            timed_ms += e0.elapsed_time(e1)
            chunks += 1
            for r in reqs:
                cache.close(r)
        calls = chunks * per_chunk
        rates[n] = {"tok_layers_per_s": n * L * calls / (timed_ms * 1e-3), "us_per_call": 1000.0 * timed_ms / calls,
                    "calls": calls, "timed_ms": timed_ms, "launches_per_call": -(-L * n // 96)}
        log(f"demote_layers batch {n}: {rates[n]['us_per_call']:.2f} us/call over {calls} calls")
        cache.close_handle()
        del cache
    del kk, vv
    rec["demote_layers"] = {"batch_1": rates[1], "batch_32": rates[32],
                            "state": f"{T0} tokens per request (64 sink + 64 history + 256 recent); chunks of "
                                     f"{per_chunk} calls timed with CUDA events, refills between chunks untimed"}
    # (2) in the fused step
    if not wl.demote_first:
        n, ra = wl.batch, wl.reqs_arr
        P = DEMOTE_STEP_PAIRS
        ptrs = [wl.pointers(s) for s in range(min(2 * P, wl.k_new.shape[0]))]
        ev = [[mk() for _ in range(6)] for _ in range(P)]
        torch.cuda.synchronize()
        for i in range(P):
            e = ev[i]
            e[0].record()
            wl.run_step(ptrs[(2 * i) % len(ptrs)], stream)
            e[1].record()
            e[2].record()
            if lib.oscar_demote_layers(wl.h, 0, L, n, ra, stream):
                raise RuntimeError(lib.oscar_last_error(wl.h).decode())
            e[3].record()
            e[4].record()
            wl.run_step(ptrs[(2 * i + 1) % len(ptrs)], stream)
            e[5].record()
        torch.cuda.synchronize()
        wl.cache.check()
        with_d = float(np.mean([1000.0 * e[0].elapsed_time(e[1]) for e in ev[1:]]))
        dl = float(np.mean([1000.0 * e[2].elapsed_time(e[3]) for e in ev[1:]]))
        without = float(np.mean([1000.0 * e[4].elapsed_time(e[5]) for e in ev[1:]]))
        rec["in_step"] = {
            "step_us_with_demote": with_d, "step_us_without_demote": without,
            "demote_cost_us_per_layer": (with_d - without) / L,
            "demote_layers_us_at_workload_state": dl,
            "demoted_tok_layers_per_s_in_steps": n * L / (with_d * 1e-6),
            "pairs": P - 1,
            "note": "whole steps (every layer's oscar_decode_step), CUDA events around each; the cost is the "
                    "difference per layer between a step whose appends demote and one whose appends find room"}
        log(f"in-step demotion: {with_d:.1f} vs {without:.1f} us/step ({(with_d - without) / L:.2f} us/layer); "
            f"demote_layers {dl:.1f} us")
    return rec


def bf16_baseline(wl, r, log, launches: int = 40):
    """Uncompressed BF16 paged decode (oscar_bf16_decode) over the same lengths, heads
    and queries, timed like the decode kernels: CUDA events around each call on the
    launching stream.  Two layers' pools alternate (each larger than L2); values are
    seeded normal bf16 (the kernel's time does not depend on them)."""
    import torch
    b = wl.b
    lens = [wl.cache.length(q, 0)[0] for q in wl.reqs]
    n, hkv = wl.batch, wl.hkv
    pages = [(t + 63) // 64 for t in lens]
    total = sum(pages)
    gen = torch.Generator(device="cuda").manual_seed(7)
    pools, tables = [], []
    for layer in range(2):
        pool = torch.randn((total, hkv, 2, 64, 128), generator=gen, device="cuda", dtype=torch.float32)
        pools.append(pool.to(torch.bfloat16))
        del pool
        perm = torch.randperm(total, generator=gen, device="cuda").to(torch.int32)
        pt = torch.zeros((n, max(pages)), dtype=torch.int32, device="cuda")
        o = 0
        for i, np_ in enumerate(pages):
            pt[i, :np_] = perm[o:o + np_]
            o += np_
        tables.append(pt)
    out = torch.empty((n, wl.hq, 128), dtype=torch.float32, device="cuda")
    ws = None
    for i in range(3):
        ws = b.bf16_decode(pools[i % 2], tables[i % 2], lens, wl.q[i, 0], out, hkv, workspace=ws)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(launches)]
    for i, (e0, e1) in enumerate(ev):
        e0.record()
        b.bf16_decode(pools[i % 2], tables[i % 2], lens, wl.q[i % wl.q.shape[0], 0], out, hkv, workspace=ws)
        e1.record()
    torch.cuda.synchronize()
    if int(ws[:4].view(torch.int32).item()) != 0:
        raise RuntimeError("bf16 baseline: page id outside the pool")
    us = float(np.mean([1000.0 * a.elapsed_time(c) for a, c in ev]))
    nbytes = sum(lens) * hkv * BF16_BYTES_PER_TOKEN_HEAD
    gbs = nbytes / (us * 1e-6) / 1e9
    int2_us = r["us_step"] / wl.L
    log(f"bf16 baseline {us:.1f} us/layer ({gbs:.0f} GB/s); INT2 step {int2_us:.1f} us/layer")
    del pools
    return {"kernel": "bf16_stream_kernel + bf16_merge_kernel (oscar_bf16_decode)", "us_per_layer": us,
            "traffic_stream_kernel": committed_traffic("bf16_stream_kernel"),
            "bytes_per_layer": nbytes, "achieved_gbs": gbs, "frac": gbs / r["peak"], "peak_source": r["peak_kind"],
            "launches_timed": launches,
            "int2_step_us_per_layer": int2_us, "speedup_of_int2_step": us / int2_us,
            "timing": "CUDA events around each call, two alternating layer pools larger than L2"}


def speedup_table(args, log):
    """INT2 cache vs the uncompressed BF16 baseline at the pages' decode shapes:
    Qwen3-8B attention (32/8 heads), contexts 30K / 60K / 100K, batch 1 and 32.
    Two layers per case, alternating (each layer's KV is read once per step, as in
    a model), CUDA events around the whole loop of K steps."""
    import torch
    rows = []
    K = max(10, min(args.steps, 40))
    for batch in (1, 32):
        for ctx in (30000, 60000, 100000):
            wl = Workload(2, args.warmup + 2 * K, log, layers=2, override={"context": ctx, "batch": batch})
            stream = wl.stream_ptr()
            ptrs = [wl.pointers(s) for s in range(args.warmup + 2 * K)]
            mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
            for s in range(args.warmup):
                wl.run_step(ptrs[s], stream)
            torch.cuda.synchronize()
            a, b = mk(), mk()
            a.record()
            for i in range(K):
                wl.run_step(ptrs[args.warmup + i], stream)
            b.record()
            torch.cuda.synchronize()
            step_us = 1000.0 * a.elapsed_time(b) / (K * wl.L)
            # decode alone (no append), same layers alternating
            lib, h, n, ra = wl.lib, wl.h, wl.batch, wl.reqs_arr
            a, b = mk(), mk()
            a.record()
            for i in range(K):
                for layer, (_, _, qp, op) in enumerate(ptrs[args.warmup + K + i]):
                    if lib.oscar_decode_attention(h, layer, n, ra, qp, op, wl.ws_ptr, wl.ws_len, stream):
                        raise RuntimeError(lib.oscar_last_error(h).decode())
            b.record()
            torch.cuda.synchronize()
            wl.cache.check()
            dec_us = 1000.0 * a.elapsed_time(b) / (K * wl.L)
            peak, kind = measured_peak_hbm()
            bf = bf16_baseline(wl, {"us_step": step_us * wl.L, "peak": peak, "peak_kind": kind}, log, launches=K)
            int2_bytes = np.mean([wl.decode_bytes(layer) for layer in range(wl.L)])
            rows.append({"context": ctx, "batch": batch, "int2_step_us": step_us, "int2_decode_us": dec_us,
                         "int2_decode_gbs": int2_bytes / (dec_us * 1e-6) / 1e9, "bf16_decode_us": bf["us_per_layer"],
                         "bf16_gbs": bf["achieved_gbs"], "speedup_step": bf["us_per_layer"] / step_us,
                         "speedup_decode": bf["us_per_layer"] / dec_us})
            log(json.dumps(rows[-1]))
            del wl
            torch.cuda.empty_cache()
    return {"table": "int2_vs_bf16_decode_per_layer", "model": "Qwen3-8B attention shape (32 q / 8 kv heads, d 128)",
            "layers_alternated": 2, "steps": K, "warmup": args.warmup, "peak_gbs": measured_peak_hbm()[0],
            "rows": rows,
            "note": "us per layer; step = oscar_decode_step (append with demote + decode); decode = "
                    "oscar_decode_attention alone; bf16 = oscar_bf16_decode over the same lengths"}


# ----------------------------------------------------------------------------------------------
PREFILL_FLOP_PER_TOKEN_HEAD = 2 * 2 * 128 * 128      # K and V rotation, one multiply-add = 2 flops


def run_write(args, log):
    """Qwen3-8B write path: prefill-quantize of a 32768-token prompt per layer, then
    single-token appends (each demoting the oldest recent token) for every layer."""
    import torch
    from bit_rotated_kv_decode_gb300 import binding, build, calibrate, synth
    build.build()
    rank, world, local = dist_info()
    torch.cuda.set_device(local)
    w = WORKLOADS[args.config]
    L = args.layers or w["layers"]
    hq, hkv, T = w["q_heads"], w["kv_heads"], w["context"]
    W, K = args.warmup, args.steps
    n_app = W + K + 4
    rk, rv, tk, tv = calibrate.calibrate_model(args.config, L, hq, hkv)
    max_pages = pages_for(T + n_app + 64) + 1
    cfg = binding.make_config(L, hq, hkv, 1, max_pages, max_pages + 8, 0, 0.0, synth.seed_for(args.config, 0, 0, 99) or 1)
    cache = binding.OscarCache(cfg, torch.from_numpy(rk).cuda(), torch.from_numpy(rv).cuda(), tk, tv)
    r = cache.open()
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    pre_us = []
    for layer in range(L):
        k = synth.kv_tokens(args.config, layer, hkv, "k", range(0, T), device="cuda")
        v = synth.kv_tokens(args.config, layer, hkv, "v", range(0, T), device="cuda")
        torch.cuda.synchronize()
        a, b = mk(), mk()
        a.record()
        cache.prefill(r, layer, k, v)
        b.record()
        torch.cuda.synchronize()
        pre_us.append(1000.0 * a.elapsed_time(b))
        del k, v
    cache.check()
    kn = torch.stack([synth.kv_tokens(args.config, l, hkv, "k", range(T, T + n_app), device="cuda", stream_id=7)
                      for l in range(L)], 1)            # [step][layer][Hkv][128]
    vn = torch.stack([synth.kv_tokens(args.config, l, hkv, "v", range(T, T + n_app), device="cuda", stream_id=7)
                      for l in range(L)], 1)
    lib, h = cache.lib, cache.h
    ra = (ctypes.c_int32 * 1)(r)
    stream = torch.cuda.current_stream().cuda_stream

    def step(s):
        for layer in range(L):
            if lib.oscar_append(h, layer, 1, ra, kn[s, layer].data_ptr(), vn[s, layer].data_ptr(), stream):
                raise RuntimeError(lib.oscar_last_error(h).decode())

    for s in range(W):
        step(s)
    torch.cuda.synchronize()
    a, b = mk(), mk()
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        a.record()
        for s in range(W, W + K):
            step(s)
        b.record()
        torch.cuda.synchronize()
        barrier(world)
    cache.check()
    ms = max_over_ranks(a.elapsed_time(b), world)
    tok_s = world * K * L / (ms * 1e-3)
    # end to end: each step's new k / v copied from pinned host memory, the error word read back
    khost, vhost = kn[W + K:].cpu().pin_memory(), vn[W + K:].cpu().pin_memory()
    e0, e1 = mk(), mk()
    torch.cuda.synchronize()
    e0.record()
    for i in range(khost.shape[0]):
        kn[W + K + i].copy_(khost[i], non_blocking=True)
        vn[W + K + i].copy_(vhost[i], non_blocking=True)
        step(W + K + i)
    e1.record()
    cache.check()
    e2e_tok_s = khost.shape[0] * L / (e0.elapsed_time(e1) * 1e-3)
    pre_avg = float(np.mean(pre_us[1:] if len(pre_us) > 1 else pre_us))
    flops = (T - 320) * hkv * PREFILL_FLOP_PER_TOKEN_HEAD
    achieved = flops / (pre_avg * 1e-6) / 1e12
    peak, peak_src = measured_peak_bf16()
    hbm_peak, hbm_src = measured_peak_hbm()
    pre_bytes = T * hkv * 512 + (T - 320) * hkv * INT2_BYTES_PER_TOKEN_HEAD + 320 * hkv * 512
    return {
        "metric": METRIC, "value": tok_s, "unit": "demoted tok/s (tokens x layers / s)", "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp32", "data": "synthetic",
        "config": {"workload": w["name"], "layers": L, "kv_heads": hkv, "head_dim": 128, "batch": 1, "context": T,
                   "step": "one oscar_append per layer (each demotes the oldest recent token)",
                   "l2": "prefill reads %.0f MB per layer from inputs larger than L2; appends touch a few KB"
                         % (pre_bytes / 1e6)},
        "prefill_us_per_layer": pre_avg,
        "prefill_gbs": pre_bytes / (pre_avg * 1e-6) / 1e9,
        # the prefill moves 154 MB per layer against 17 GFLOP of rotation: HBM is the bound
        "roofline": {"bound": "hbm", "kernel": "prefill (prefill_hist_kernel + prefill_bf16_kernel, one call)",
                     "achieved": pre_bytes / (pre_avg * 1e-6) / 1e9, "peak": hbm_peak, "unit": "GB/s",
                     "frac": pre_bytes / (pre_avg * 1e-6) / 1e9 / hbm_peak, "peak_source": hbm_src,
                     "bytes": "algorithmic per layer: every token's bf16 K and V read, the history's INT2 codes "
                              "and meta and the BF16 segments written",
                     "algorithmic_bytes_per_launch": pre_bytes,
                     "duration_us_per_launch": pre_avg,
                     "duration_from": "CUDA events around each layer's oscar_prefill_quantize call",
                     "traffic": committed_traffic("prefill_hist_kernel"),
                     "traffic_kernel": "prefill_hist_kernel",
                     "tensor": {"achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                                "peak_source": peak_src,
                                "flops": "algorithmic: 2 x 128 x 128 per token, kv head and K or V"}},
        "e2e": {"value": e2e_tok_s, "unit": "demoted tok/s (tokens x layers / s)",
                "h2d_bytes_per_step": (kn[0].numel() + vn[0].numel()) * 2, "d2h_bytes_per_step": 4},
        "gpu_launches": K * L,
        "clocks": clk.summary(),
    }


# ----------------------------------------------------------------------------------------------
def oracle_inputs(wl, layer: int):
    """Host float64 K / V of request 0 of one layer at the cache's current state."""
    import torch
    hkv = wl.hkv
    r = wl.reqs[0]
    t, he = wl.cache.length(r, layer)
    t0 = wl.lens[0]
    n_new = t - t0
    parts_k, parts_v = [], []
    if wl.prefix:
        gen = lambda which: wl.synth.kv_tokens(wl.cfg_id, layer, hkv, which, range(0, wl.prefix + 256),  # noqa: E731
                                               total_len=wl.prefix + 256, drift=wl.drift, device="cuda",
                                               stream_id=0)[:wl.prefix]
        parts_k.append(gen("k"))
        parts_v.append(gen("v"))
    p0 = wl.prefix
    parts_k.append(wl.synth.kv_tokens(wl.cfg_id, layer, hkv, "k", range(p0, t0), total_len=t0, drift=wl.drift,
                                      device="cuda", stream_id=wl.sid[0]))
    parts_v.append(wl.synth.kv_tokens(wl.cfg_id, layer, hkv, "v", range(p0, t0), total_len=t0, drift=wl.drift,
                                      device="cuda", stream_id=wl.sid[0]))
    k = torch.cat(parts_k + [wl.k_new[:n_new, layer, 0]]).float().cpu().numpy().astype(np.float64)
    v = torch.cat(parts_v + [wl.v_new[:n_new, layer, 0]]).float().cpu().numpy().astype(np.float64)
    return k, v, t, he


def cpu_baseline(wl, res, log):
    """Time the oracle on the host cores for layer 0 of request 0 and check the GPU output there."""
    import torch
    from oracle import attention
    from tests import parity
    layer = 0
    k, v, t, he = oracle_inputs(wl, layer)
    # recompute layer 0's decode on the GPU at this exact state and compare
    q = wl.q[0, layer].contiguous()
    out = torch.empty((wl.batch, wl.hq, 128), dtype=torch.float32, device="cuda")
    wl.cache.decode(layer, wl.reqs, q, out, wl.ws)
    wl.cache.check()
    qf = q[0].float().cpu().numpy().astype(np.float64)
    cores = len(os.sched_getaffinity(0))
    t0 = time.time()
    ref = attention.decode(qf, k, v, he, wl.rk[layer].astype(np.float64), wl.rv[layer].astype(np.float64),
                           wl.tk[layer], wl.tv[layer], group=wl.group)
    secs = time.time() - t0
    par = parity.check_output(out[0].cpu().numpy(), ref)
    return {
        "value": secs * 1e6 * wl.L,
        "unit": "us/step",
        "cores": cores,
        "kind": "oracle",
        "sample": f"layer {layer} of {wl.L}, request 0, all {wl.hq} query heads over {t} tokens "
                  f"(oracle quantises the history itself), extrapolated x{wl.L} layers; "
                  f"measured {secs:.2f} s for the sample",
    }, {"layer": layer, "tokens": t, "hist_end": he, **par,
        "thresholds": {"max_abs": parity.OUT_MAX_ABS, "rel_fro": parity.OUT_REL_FRO}}


# ----------------------------------------------------------------------------------------------
def run_reference(args, log):
    """The oracle as it stands, timed on the host cores on a bounded sample per step."""
    rank, world, _ = dist_info()
    if rank != 0:
        return None
    import torch
    from bit_rotated_kv_decode_gb300 import calibrate, synth
    from oracle import attention
    w = WORKLOADS[args.config]
    L, hq, hkv, T = w["layers"], w["q_heads"], w["kv_heads"], w["context"]
    g = hq // hkv
    rk, rv, tk, tv = calibrate.calibrate_model(args.config, 1, hq, hkv)
    # one kv head (its GQA group of query heads) of layer 0 per step, drawn on the host
    k = synth.kv_tokens(args.config, 0, hkv, "k", range(0, T), total_len=T).to(torch.float64).numpy()[:, :1]
    v = synth.kv_tokens(args.config, 0, hkv, "v", range(0, T), total_len=T).to(torch.float64).numpy()[:, :1]
    cores = len(os.sched_getaffinity(0))
    times = []
    for s in range(args.warmup + args.steps):
        q = synth.queries(args.config, 0, hq, 1, s).to(torch.float64).numpy()[0, :g]
        t0 = time.time()
        attention.decode(q, k, v, T - 256, rk[0, :1].astype(np.float64), rv[0, :1].astype(np.float64),
                         tk[0, :1], tv[0, :1])
        if s >= args.warmup:
            times.append(time.time() - t0)
    per_step_us = float(np.mean(times)) * 1e6 * hkv * L
    sample = (f"layer 0, kv head 0 and its {g} query heads over {T} tokens per step, "
              f"extrapolated x{hkv} kv heads x{L} layers")
    return {
        "metric": METRIC, "impl": "reference", "value": per_step_us, "unit": "us/step", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step_us / 1000.0, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w["name"], "layers": L, "q_heads": hq, "kv_heads": hkv, "batch": w["batch"],
                   "context": T},
        "cpu_baseline": {"value": per_step_us, "unit": "us/step", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": per_step_us, "unit": "us/step", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ----------------------------------------------------------------------------------------------
def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1400)   # a timed region of over a second at 100K x 32 layers
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--config", type=int, default=2, choices=sorted(WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-bf16-baseline", action="store_true",
                    help="skip the uncompressed BF16 decode comparison")
    ap.add_argument("--group", type=int, default=128, choices=[128, 64],
                    help="quantisation group size (64: two {s, z} per token-head, 2.5 bits)")
    ap.add_argument("--demote-first", action="store_true",
                    help="each step starts with one oscar_demote_layers over all layers; the per-layer steps "
                         "then only append")
    ap.add_argument("--speedup-table", action="store_true",
                    help="INT2 vs BF16 decode per layer at 30K / 60K / 100K, batch 1 and 32 (one JSON line)")
    ap.add_argument("--layers", type=int, default=0, help="fewer layers (small profiling cases only)")
    ap.add_argument("--no-demote-record", action="store_true",
                    help="skip the oscar_demote_layers rates and the in-step demotion cost")
    ap.add_argument("--separate-calls", action="store_true",
                    help="time oscar_append + oscar_decode_attention per layer instead of oscar_decode_step")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, _ = dist_info()
    log = (lambda m: print(f"[bench] {m}", file=sys.stderr, flush=True)) if rank == 0 else (lambda m: None)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if args.impl == "gb300" else "gloo")
    if args.impl == "reference":
        line = run_reference(args, log)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if args.speedup_table:
        import torch
        torch.cuda.set_device(0)
        print(json.dumps(speedup_table(args, log)), flush=True)
        return
    w = WORKLOADS[args.config]
    if w.get("write_path"):
        line = run_write(args, log)
        if rank == 0:
            print(json.dumps(line), flush=True)
        return
    wl, r = run_gpu(args, log)
    base16 = bf16_baseline(wl, r, log) if not args.no_bf16_baseline else None
    cpu = par = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu, par = cpu_baseline(wl, r, log)
    # last: its steps append tokens that reuse earlier inputs, which the oracle check above does not follow
    demote = demote_record(wl, log) if not args.no_demote_record else None
    traffic = committed_traffic("decode_kernel")
    kv_gbs = r["kv_bytes_step"] / (r["us_step"] * 1e-6) / 1e9
    line = {
        "metric": METRIC,
        "value": r["us_step"],
        "unit": "us/step",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": r["us_step"] / 1000.0,
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp32",
        "data": "synthetic",
        "config": {"workload": w["name"], "layers": wl.L, "q_heads": wl.hq, "kv_heads": wl.hkv, "head_dim": 128,
                   "batch": wl.batch,
                   "context": wl.T0 if len(set(wl.lens)) == 1 else "%d..%d (mean %d)" % (
                       min(wl.lens), max(wl.lens), int(np.mean(wl.lens))),
                   "shared_prefix_tokens": wl.prefix, "page_tokens": 64, "page_order": "seeded shuffle",
                   "storage": "INT2 codes + fp16 scale/zero history, BF16 sink/recent",
                   "quant_group": wl.group,
                   "step": (("oscar_demote_layers over all layers, then " if args.demote_first else "") +
                            ("per layer: oscar_decode_step (append" +
                             (", then decode attention)" if args.demote_first else
                              " with fused demote, then decode attention)")
                             if not args.separate_calls else
                             "per layer: oscar_append" + ("" if args.demote_first else " (fused demote)") +
                             " then oscar_decode_attention")),
                   "l2": "inputs larger than L2 (%.2f GB of KV per step vs 129 MB L2)" % (
                       r["bytes_per_launch"] * wl.L / 1e9),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "kv_gbs_step": kv_gbs,
        "decode_bytes_per_layer_logical": wl.decode_bytes(0, unique=False),
        "kv_frac_of_8tbs_step": kv_gbs / NOMINAL_HBM_GBS,
        "decode_us_per_layer": r["dec_avg_us"],
        "append_us_per_layer": r["app_avg_us"],
        "demote_tok_s": None if args.demote_first else wl.batch * 1e6 / r["app_avg_us"],
        "roofline": {"bound": "hbm", "kernel": "decode_kernel", "achieved": r["achieved_gbs"], "peak": r["peak"],
                     "unit": "GB/s", "frac": r["achieved_gbs"] / r["peak"], "peak_source": r["peak_kind"],
                     "traffic": traffic, "algorithmic_bytes_per_launch": r["bytes_per_launch"],
                     "duration_us_per_launch": r["launch_us"],
                     "duration_from": ("timed region / (steps x layers): one oscar_decode_step per layer "
                                       "(append + stream + merge in one kernel), an upper bound on the kernel's time"
                                       if not args.separate_calls else
                                       "CUDA events around each oscar_decode_attention call")},
        "e2e": {"value": r["e2e_us"], "unit": "us/step", "h2d_bytes_per_step": r["h2d"],
                "d2h_bytes_per_step": r["d2h"],
                "copies": "pinned host buffers, inputs and outputs on their own streams overlapping the neighbouring steps"},
        "gpu_launches": r["launches"],
        "clocks": r["clocks"],
    }
    if base16 is not None:
        line["bf16_baseline"] = base16
    if demote is not None:
        line["demote"] = demote
    if cpu is not None:
        line["cpu_baseline"] = cpu
        line["parity"] = par
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
