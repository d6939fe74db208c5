"""Byte and flop accounting of bench.py, checked against the layout on the host.

The roofline's `achieved` divides algorithmic bytes by a measured time; these
tests pin the byte counts to the record layout (oracle/layout.py) and to the
100K workload's figures, so a wrong count cannot inflate or deflate it.
"""
import bench
from oracle import layout


def test_int2_bytes_per_token_head_follow_the_record():
    for group in (128, 64):
        rec = layout.record_layout(group)["record"]
        assert bench.int2_bytes_per_token_head(group) * layout.PAGE_TOKENS == rec
    assert bench.int2_bytes_per_token_head() == bench.INT2_BYTES_PER_TOKEN_HEAD == 72
    assert bench.BF16_BYTES_PER_TOKEN_HEAD == 2 * 128 * 2


def test_decode_bytes_at_100k():
    # 100,000 tokens: 64 sink, 256 recent, 99,680 INT2 history, 8 kv heads
    assert bench.algorithmic_bytes(100000, 100000 - 256, 8) == 99680 * 8 * 72 + 320 * 8 * 512 == 58726400
    assert bench.algorithmic_bytes(100000, 100000 - 256, 8, group=64) == 99680 * 8 * 80 + 320 * 8 * 512


def test_decode_bytes_short_requests():
    # all sink; sink plus part of the window; nothing demoted yet
    assert bench.algorithmic_bytes(30, 64, 8) == 30 * 8 * 512
    assert bench.algorithmic_bytes(200, 64, 8) == 200 * 8 * 512
    assert bench.algorithmic_bytes(321, 65, 8) == 1 * 8 * 72 + 320 * 8 * 512


def test_history_pages():
    assert bench.pages_for(64) == 0 and bench.pages_for(65) == 1 and bench.pages_for(128) == 1
    assert bench.pages_for(129) == 2
    assert bench.pages_for(100000 - 256) == (99680 + 63) // 64


def test_prefill_flops():
    # rotation of K and V: one 128 x 128 matrix-vector product each, 2 flops per multiply-add
    assert bench.PREFILL_FLOP_PER_TOKEN_HEAD == 2 * 2 * 128 * 128
