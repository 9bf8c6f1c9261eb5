"""Algorithmic byte counts used by the roofline figures, against sizes worked
out by hand from the layouts (and, for the 397B expert, the size the flash-moe
article gives in "SSD Expert Streaming": about 6.75 MB per 4-bit expert)."""
import json
import os

import synth
from quantized_moe_decode_layer_gb300.accounting import expert_bytes, layer_flops, row_bytes, unique_bytes

HERE = os.path.dirname(os.path.abspath(__file__))


def test_row_bytes():
    assert row_bytes(2048, 6) == 1536 + 32 * 4
    assert row_bytes(512, 6) == 384 + 8 * 4
    assert row_bytes(2048, 8) == 2048 + 32 * 4
    assert row_bytes(256, 0) == 1024


def test_expert_bytes_match_page_size():
    gold = json.load(open(os.path.join(HERE, "golden", "page_sizes.json")))
    assert expert_bytes(4096, 1024, 4) == 7_077_888
    assert abs(expert_bytes(4096, 1024, 4) / 2 ** 20 - 6.75) < 1e-12
    assert any(abs(v - 6.75) < 1e-9 for v in _numbers(gold))


def _numbers(d):
    if isinstance(d, dict):
        for v in d.values():
            yield from _numbers(v)
    elif isinstance(d, list):
        for v in d:
            yield from _numbers(v)
    elif isinstance(d, (int, float)):
        yield d


def test_unique_bytes_by_hand():
    # a35b at M=1: 8 experts of 2*512*1664 + 2048*416 bytes, the 8-bit shared
    # expert 2*512*2176 + 2048*544, 257 router rows of 2176, two bf16 gammas,
    # x / out / out_n rows of 4096 bytes
    a = 8 * (2 * 512 * 1664 + 2048 * 416) + (2 * 512 * 2176 + 2048 * 544) + 257 * 2176 + 2 * 4096 + 3 * 4096
    assert a == 24_369_280
    assert unique_bytes(synth.A35B, 8, 1) == a
    assert unique_bytes(synth.A35B, 18, 4) == 18 * 2_555_904 + 3_958_912
    assert unique_bytes(synth.B397, 10, 1) == 86_421_760
    # tiny: fp32 router, no shared expert, 4-bit experts of 2*128*144 + 256*72
    assert unique_bytes(synth.TINY, 2, 1) == 2 * (2 * 128 * 144 + 256 * 72) + 16 * 1024 + 2 * 512 + 3 * 512


def test_flops():
    assert layer_flops(synth.A35B, 8, 1) == 8 * 6 * 512 * 2048 + 6 * 512 * 2048 + 2 * 257 * 2048


def test_traffic_record_scales_with_layers():
    """The bench's DRAM-traffic figure is per launch of the stack it ran: the
    committed record (40 layers) scales with the launch's layer count."""
    import bench
    rec = {"bytes_per_launch": 992006827, "layers": 40}
    assert bench.traffic_for(rec, 40) == 992006827
    assert bench.traffic_for(rec, 8) == round(992006827 * 8 / 40)
    assert bench.traffic_for(None, 8) is None
