"""Byte layout of the three-segment cache (oracle; test infrastructure).

[MTP] section "The Serving System: Mixed-Precision Cache Layout": per request a
BF16 sink of the first S0 = 64 tokens, a BF16 window of the last W = 256
tokens, INT2 history in between, paged like a standard paged KV cache.
[MS] section "OSCAR的设计": four 2-bit values are packed into one byte.

Readings (the pages give no byte layout):
  * a page holds 64 tokens; one INT2 page-head record is 4608 bytes:
      [   0, 2048) K codes, token slot r at r*32 (32 bytes = 128 codes)
      [2048, 4096) V codes, same layout
      [4096, 4352) K meta, slot r at 4096 + 4r: fp16 s then fp16 z
      [4352, 4608) V meta, same layout
    i.e. 72 bytes = 2.25 bits per element per token-head;
  * with G_K = 64 (two groups per token-head) the record is 5120 bytes: codes
    as above, then K meta [4096, 4608) with slot r at 4096 + 8r holding group
    0's fp16 s, z then group 1's, and V meta [4608, 5120) the same way; 80
    bytes = 2.5 bits per element per token-head;
  * codes in the rotated channel order, channel 4j+i in bits 2i..2i+1 of byte j;
  * BF16 pages hold [2][64][128] bf16 per head (K rows then V rows); the
    recent window is a ring: position p >= 64 lives in ring slot (p-64) mod 256,
    i.e. ring page slot//64, row slot%64; sink position p < 64 in sink row p.
"""
from __future__ import annotations

import numpy as np

HEAD_DIM = 128
PAGE_TOKENS = 64
SINK_TOKENS = 64
RECENT_TOKENS = 256
RING_PAGES = RECENT_TOKENS // PAGE_TOKENS
CODE_BYTES = HEAD_DIM // 4          # 32 bytes of codes per token-head
META_BYTES = 4                      # fp16 s, fp16 z
K_CODES_OFF = 0
V_CODES_OFF = PAGE_TOKENS * CODE_BYTES
K_META_OFF = 2 * PAGE_TOKENS * CODE_BYTES
V_META_OFF = K_META_OFF + PAGE_TOKENS * META_BYTES
RECORD_BYTES = V_META_OFF + PAGE_TOKENS * META_BYTES   # 4608
BF16_RECORD_ELEMS = 2 * PAGE_TOKENS * HEAD_DIM         # K rows then V rows


def record_layout(group: int = 128) -> dict:
    """Offsets of one page-head record for a quantisation group size (128 or 64)."""
    if group not in (64, 128):
        raise ValueError("group size must be 64 or 128")
    meta = META_BYTES * (HEAD_DIM // group)
    k_meta = 2 * PAGE_TOKENS * CODE_BYTES
    v_meta = k_meta + PAGE_TOKENS * meta
    return {"k_codes": K_CODES_OFF, "v_codes": V_CODES_OFF, "k_meta": k_meta, "v_meta": v_meta,
            "meta_bytes": meta, "record": v_meta + PAGE_TOKENS * meta}


def pack_codes(codes: np.ndarray) -> np.ndarray:
    """uint8 [..., 128] codes in 0..3 -> uint8 [..., 32] packed bytes."""
    c = codes.astype(np.uint32).reshape(codes.shape[:-1] + (HEAD_DIM // 4, 4))
    b = np.zeros(c.shape[:-1], dtype=np.uint32)
    for i in range(4):
        b |= c[..., i] << (2 * i)
    return b.astype(np.uint8)


def unpack_codes(packed: np.ndarray) -> np.ndarray:
    """uint8 [..., 32] -> uint8 [..., 128]."""
    p = packed.astype(np.uint32)
    out = np.zeros(packed.shape[:-1] + (packed.shape[-1], 4), dtype=np.uint8)
    for i in range(4):
        out[..., i] = (p >> (2 * i)) & 3
    return out.reshape(packed.shape[:-1] + (packed.shape[-1] * 4,))


def meta_bytes(s: np.ndarray, z: np.ndarray, groups: int = 1) -> np.ndarray:
    """uint8 [..., 4 * groups]: per group, little-endian fp16 s then fp16 z.

    With groups > 1, s and z carry a trailing [groups] axis."""
    s16 = np.asarray(s, dtype=np.float16).view(np.uint16).astype(np.uint32)
    z16 = np.asarray(z, dtype=np.float16).view(np.uint16).astype(np.uint32)
    if groups == 1:
        s16, z16 = s16[..., None], z16[..., None]
    out = np.zeros(np.shape(s16) + (4,), dtype=np.uint8)
    out[..., 0] = s16 & 0xFF
    out[..., 1] = s16 >> 8
    out[..., 2] = z16 & 0xFF
    out[..., 3] = z16 >> 8
    return out.reshape(out.shape[:-2] + (4 * out.shape[-2],))


def record_slot_fields(record: np.ndarray, slot: int, group: int = 128):
    """Split one page-head record at token slot -> (kc, vc, kmeta, vmeta): the
    slot's packed K and V codes (32 bytes each) and its K and V meta bytes."""
    lay = record_layout(group)
    mb = lay["meta_bytes"]
    kc = record[K_CODES_OFF + slot * CODE_BYTES: K_CODES_OFF + (slot + 1) * CODE_BYTES]
    vc = record[V_CODES_OFF + slot * CODE_BYTES: V_CODES_OFF + (slot + 1) * CODE_BYTES]
    km = record[lay["k_meta"] + slot * mb: lay["k_meta"] + (slot + 1) * mb]
    vm = record[lay["v_meta"] + slot * mb: lay["v_meta"] + (slot + 1) * mb]
    return kc, vc, km, vm


def meta_to_sz(meta4: np.ndarray):
    """uint8 [..., 4] -> (s, z) float16 [...]; uint8 [..., 4 g] -> (s, z) [..., g]."""
    m = meta4.astype(np.uint16)
    groups = m.shape[-1] // 4
    m = m.reshape(m.shape[:-1] + (groups, 4))
    s = (m[..., 0] | (m[..., 1] << 8)).astype(np.uint16).view(np.float16)
    z = (m[..., 2] | (m[..., 3] << 8)).astype(np.uint16).view(np.float16)
    if groups == 1:
        s, z = s[..., 0], z[..., 0]
    return s, z


def ring_slot(p: int) -> int:
    """Ring slot of a recent-window position p >= 64."""
    return (p - SINK_TOKENS) % RECENT_TOKENS


def bits_per_element(total_tokens: int, group: int = 128) -> float:
    """Average stored bits per KV element of a request of ``total_tokens``.

    BF16 (16 bits) for the sink and recent windows, 2 bits of code plus 32 bits
    of fp16 (s, z) per group of ``group`` channels for history.
    """
    bf16 = min(total_tokens, SINK_TOKENS + RECENT_TOKENS)
    hist = total_tokens - bf16
    hist_bits = 2.0 + 8.0 * META_BYTES / group
    return (bf16 * 16.0 + hist * hist_bits) / total_tokens
