"""The bench's FLOP/byte accounting against the figures the pages print."""

import math

from exact_attention_84_gb300 import accounting as acc
from oracle_pins import read_golden


def test_standard_attention_traffic_matches_page():
    g = read_golden("hbm_traffic.txt")
    n, d, e = int(g["std_n"]), int(g["std_d"]), int(g["std_bytes_per_elem"])
    per_head = acc.standard_attention_hbm_elements(n, d) * e
    assert round(per_head / 1e6) == g["std_traffic_mb"]
    assert round(n * n * e / 1e6, 1) == g["std_s_mb"]
    layer_ms = 32 * per_head / 2e12 * 1e3
    assert round(layer_ms, 2) == g["std_layer_ms_at_2tbps"]


def test_io_complexity_matches_page():
    g = read_golden("hbm_traffic.txt")
    n, d, m = int(g["io_n"]), int(g["io_d"]), int(g["io_m_elems"])
    std = acc.standard_hbm_accesses(n, d)
    fl = acc.flash_hbm_accesses(n, d, m)
    assert round(std / 1e6, 1) == g["io_standard_M"]
    assert round(fl / 1e6, 1) == g["io_flash_M"]
    assert round(std / fl, 1) == g["io_ratio"]
    assert round(n * n * 2 / 1e6) == g["io_extra_scores_mb"]
    assert round(2 * n * 4 / 1e3) == g["io_extra_stats_kb"]


def test_flop_conventions():
    f = acc.forward_flops(1, 32, 8192, 128, causal=False)
    assert f == 4 * 32 * 8192 ** 2 * 128
    assert acc.forward_flops(1, 32, 8192, 128, causal=True) == f / 2
    assert acc.backward_flops(8, 32, 4096, 128, True) == 2.5 * acc.forward_flops(8, 32, 4096,
                                                                                   128, True)
    assert math.isclose(acc.decode_kv_bytes(64, 32, 32768, 128), 34.359738368e9)


def test_visible_pairs_brute_force():
    """The closed form of the visible (query, key) count against a direct
    count of the mask."""
    for n in (1, 5, 17, 64):
        for causal, window in ((False, 0), (True, 0), (True, 1), (True, 3), (True, 16),
                               (True, 100)):
            count = sum(1 for i in range(n) for j in range(n)
                        if (not causal or j <= i) and (not window or j > i - window))
            assert acc.visible_pairs(n, causal, window) == count
