"""Cache state machine mirror (oracle; test infrastructure).

Follows the pages' runtime statement ([MS] section "OSCAR的设计"): a new token
is written into the BF16 recent window; as decoding advances the oldest
recent token is rotated, clipped, quantised and packed into INT2 history.

State of one (request, layer): T tokens cached, hist_end = end of the INT2
history (history = [64, hist_end), recent = [hist_end, T)).  Readings:
  * append of position p = T: p < 64 goes to sink row p; otherwise, when the
    recent window already holds 256 tokens, token hist_end is demoted first
    (its ring slot is the new token's slot), then the new token is written
    to ring slot (p - 64) mod 256;
  * demote: the oldest recent token goes to history (window shrinks by one);
  * prefill of n tokens on an empty request (or one whose recent window is
    empty) equals n appends;
  * fork(parent, P): P >= 64, (P - 64) % 64 == 0, and in every layer the
    parent has already demoted every position below P; the child shares the
    sink page and the history pages of positions 64..P-1 and starts with
    T = hist_end = P;
  * history page index i of a request is allocated when a layer first writes
    history token 64 + 64 i; the page table is shared by all layers;
  * request ids are the lowest free slot; open takes one sink and four ring
    BF16 pages (a fork takes four ring pages and shares the sink); close
    releases history pages in index order, then the sink, then the ring pages.
Expected bytes are a function of the token sequence alone because every token
is quantised on its own (one group per token-head).
"""
from __future__ import annotations

import numpy as np

from . import layout, quant
from .alloc import PagePool

SINK = layout.SINK_TOKENS
W = layout.RECENT_TOKENS
P = layout.PAGE_TOKENS


class StateError(Exception):
    pass


class Request:
    def __init__(self, num_layers: int):
        self.hist_pt: list[int] = []
        self.bf16_pt: list[int] = []          # [sink, ring0..ring3]
        self.T = [0] * num_layers
        self.hist_end = [SINK] * num_layers


class CacheMirror:
    def __init__(self, num_layers: int, num_kv_heads: int, max_requests: int, max_pages_per_request: int,
                 num_int2_pages: int, num_bf16_pages: int, page_perm_seed: int = 0):
        self.L = num_layers
        self.hkv = num_kv_heads
        self.max_requests = max_requests
        self.max_pages = max_pages_per_request
        self.int2 = PagePool(num_int2_pages, page_perm_seed)
        self.bf16 = PagePool(num_bf16_pages, 0)
        self.reqs: dict[int, Request] = {}

    # -- requests ---------------------------------------------------------
    def _slot(self) -> int:
        for i in range(self.max_requests):
            if i not in self.reqs:
                return i
        raise StateError("no free request slot")

    def open(self) -> int:
        rid = self._slot()
        if self.bf16.free_count < 1 + layout.RING_PAGES:
            raise MemoryError("out of bf16 pages")
        r = Request(self.L)
        r.bf16_pt = [self.bf16.alloc() for _ in range(1 + layout.RING_PAGES)]
        self.reqs[rid] = r
        return rid

    def fork(self, parent: int, prefix: int) -> int:
        par = self.reqs[parent]
        if prefix < SINK or (prefix - SINK) % P != 0:
            raise StateError("prefix must be 64 + a multiple of 64")
        if any(par.hist_end[l] < prefix for l in range(self.L)):
            raise StateError("parent has not demoted the whole prefix")
        rid = self._slot()
        if self.bf16.free_count < layout.RING_PAGES:
            raise MemoryError("out of bf16 pages")
        r = Request(self.L)
        self.bf16.share(par.bf16_pt[0])
        r.bf16_pt = [par.bf16_pt[0]] + [self.bf16.alloc() for _ in range(layout.RING_PAGES)]
        npages = (prefix - SINK) // P
        for i in range(npages):
            self.int2.share(par.hist_pt[i])
        r.hist_pt = list(par.hist_pt[:npages])
        r.T = [prefix] * self.L
        r.hist_end = [prefix] * self.L
        self.reqs[rid] = r
        return rid

    def close(self, rid: int) -> None:
        r = self.reqs.pop(rid)
        for p in r.hist_pt:
            self.int2.release(p)
        for p in r.bf16_pt:
            self.bf16.release(p)

    # -- writes -----------------------------------------------------------
    def _ensure_page(self, r: Request, h: int) -> None:
        """Allocate, in index order, every missing page up to the one of history index h."""
        while len(r.hist_pt) <= h // P:
            r.hist_pt.append(self.int2.alloc())

    def _check_room(self, r: Request, h_end: int) -> None:
        if h_end > SINK and (h_end - SINK + P - 1) // P > self.max_pages:
            raise StateError("request exceeds its page table")
        if self._pages_needed(r, h_end) > self.int2.free_count:
            raise MemoryError("out of pages")

    def _pages_needed(self, r: Request, h_end: int) -> int:
        if h_end <= SINK:
            return 0
        need = (h_end - SINK + P - 1) // P
        return max(0, need - len(r.hist_pt))

    def append(self, rid: int, layer: int) -> dict:
        """Advance (rid, layer) by one token; returns what the kernel must do."""
        r = self.reqs[rid]
        p = r.T[layer]
        act = {"pos": p, "demote": None}
        if p >= SINK and p - r.hist_end[layer] == W:
            self._check_room(r, r.hist_end[layer] + 1)
            act["demote"] = r.hist_end[layer]
            self._ensure_page(r, r.hist_end[layer] - SINK)
            r.hist_end[layer] += 1
        r.T[layer] = p + 1
        return act

    def demote(self, rid: int, layer: int) -> int:
        r = self.reqs[rid]
        if r.T[layer] <= SINK or r.hist_end[layer] >= r.T[layer]:
            raise StateError("recent window is empty")
        self._check_room(r, r.hist_end[layer] + 1)
        h = r.hist_end[layer]
        self._ensure_page(r, h - SINK)
        r.hist_end[layer] += 1
        return h

    def prefill(self, rid: int, layer: int, n: int) -> None:
        r = self.reqs[rid]
        t0 = r.T[layer]
        if not (t0 == 0 or (t0 >= SINK and r.hist_end[layer] == t0)):
            raise StateError("prefill needs an empty recent window")
        total = t0 + n
        new_hist_end = max(r.hist_end[layer], total - W, SINK)
        self._check_room(r, new_hist_end)
        if new_hist_end > r.hist_end[layer]:
            self._ensure_page(r, new_hist_end - 1 - SINK)
        r.hist_end[layer] = new_hist_end
        r.T[layer] = total


def expected_history(k_head: np.ndarray, v_head: np.ndarray, rk: np.ndarray, rv: np.ndarray,
                     tau_k: float, tau_v: float, group: int = 128):
    """Codes / meta of history tokens of one head (rows of k_head, v_head).

    Returns dict of packed K/V code bytes [n][32], meta bytes [n][4 * groups],
    the raw codes, s, z and the fp32 rotated values (for exemption bands).
    """
    ck, sk, zk, xk = quant.quantize_tokens(k_head, rk, np.float32(tau_k), group)
    cv, sv, zv, xv = quant.quantize_tokens(v_head, rv, np.float32(tau_v), group)
    ng = layout.HEAD_DIM // group
    return {
        "k_packed": layout.pack_codes(ck), "v_packed": layout.pack_codes(cv),
        "k_meta": layout.meta_bytes(sk, zk, ng), "v_meta": layout.meta_bytes(sv, zv, ng),
        "k_codes": ck, "v_codes": cv, "k_s": sk, "k_z": zk, "v_s": sv, "v_z": zv,
        "k_x32": xk, "v_x32": xv,
    }
