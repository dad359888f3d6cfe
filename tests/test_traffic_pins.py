"""Pins of the oracle's byte/FLOP counter against every number the pages print."""
import math

import pytest

from oracle import traffic as T

from conftest import read_golden

MIB, GIB = T.MIB, T.GIB


def _kv(name):
    return {r[0]: r[1:] for r in read_golden(name)}


def test_page1_one_head_8k():
    g = {k: float(v[0]) for k, v in _kv("page1_one_head_8k.txt").items()}
    n, d = int(g["n"]), int(g["d"])
    assert T.tensor_bytes(n, d) == g["one_tensor_mib"] * MIB
    assert T.compulsory_bytes(n, n, d) == g["compulsory_mib"] * MIB
    assert T.naive_score_bytes(n, n) == g["score_matrix_mib"] * MIB
    assert 4 * T.naive_score_bytes(n, n) == g["score_traffic_mib"] * MIB
    naive = T.naive_traffic_bytes(n, n, d)
    assert naive == g["naive_total_mib"] * MIB
    assert round(T.seconds(naive, 3.35e12) * 1e6) == g["naive_time_us_at_3.35TBps"]
    assert n // 128 == g["paper_blocks_br128"]
    assert (n // 128) * 2 * T.tensor_bytes(n, d) == g["paper_kv_reads_mib_br128"] * MIB
    assert T.paper_model_bytes(n, d, 128) == g["paper_total_mib_br128"] * MIB
    assert T.paper_model_bytes(n, d, 64) == g["paper_total_mib_br64"] * MIB
    comp = T.compulsory_bytes(n, n, d)
    assert round(comp / 1e4) * 1e4 == g["real_hbm_bytes"]
    fl = T.forward_flops(n, n, d)
    assert round(fl / 1e8) / 10 == g["flops_gflop"]
    assert T.intensity(fl, comp) == g["intensity_flop_per_byte"]
    assert round(989e12 / 3.35e12) == g["h100_ridge_flop_per_byte"]
    assert round(T.seconds(fl, 989e12) * 1e7) / 10 == g["compute_time_us_at_989TFLOPs"]
    assert round(T.seconds(comp, 3.35e12) * 1e7) / 10 == g["hbm_time_us_at_3.35TBps"]
    assert naive / comp == g["naive_over_real"]
    assert round(T.forward_flops(n, n, d, causal=True) / 1e8) / 10 == g["causal_flops_gflop"]
    assert T.decode_kv_bytes_per_kv_head(n, d) == g["decode_kv_mib_per_kv_head"] * MIB
    # one query head per KV head: 4 N d FLOPs over the 4 N d bytes of K and V
    assert (T.decode_flops_per_query_head(n, d) / T.decode_kv_bytes_per_kv_head(n, d)
            == g["decode_flop_per_byte_per_group_member"])
    # a GQA group of 4 query heads on one KV head: intensity x4
    assert (4 * T.decode_flops_per_query_head(n, d) / T.decode_kv_bytes_per_kv_head(n, d)) == 4.0


def test_page2_footprint_and_score_tables():
    for row in read_golden("page2_tables.txt"):
        if row[0] == "footprint":
            n = int(row[1])
            std = T.standard_footprint_bytes(n, 32, 128) / MIB
            fl = T.flash_footprint_bytes(n, 32, 128) / MIB
            assert f"{std:.1f}" == row[2]
            assert f"{fl:.1f}" == row[3]
            assert f"{std / fl:.1f}" == row[4]
            assert f"{std - fl:.1f}" == row[5]
        elif row[0] == "score":
            n = int(row[1])
            assert f"{32 * T.naive_score_bytes(n, n) / GIB:.2f}" == row[2]


def test_page2_sram_table_and_block_rule():
    for row in read_golden("page2_tables.txt"):
        if row[0] == "sram":
            b = int(row[1])
            assert f"{b * 128 * 2 / 1024:.1f}" == row[2]
            assert f"{2 * b * 128 * 2 / 1024:.1f}" == row[3]
            assert f"{b * 128 * 2 / 1024:.1f}" == row[4]
            assert f"{b * 2 * 4 / 1024:.1f}" == row[5]
            tot = T.sram_tile_bytes(b, 128) / 1024
            assert f"{tot:.1f}" == row[6]
            assert ("YES" if tot <= 192 else "NO") == row[7]
            assert f"{T.tile_intensity(b, 128):.1f}" == row[8]
        elif row[0] == "best":
            kb, blk, ai = int(row[1]), int(row[2]), float(row[3])
            assert T.best_block(kb * 1024, 128) == blk
            assert T.tile_intensity(blk, 128) == ai


def test_page2_traffic_table_and_context():
    for row in read_golden("page2_tables.txt"):
        if row[0] == "traffic":
            n = int(row[1])
            std = T.standard_traffic_bytes(n, 32, 128)
            fl = T.flash_traffic_bytes(n, 32, 128)
            assert f"{std / GIB:.2f}" == row[2]
            assert f"{fl / GIB:.3f}" == row[3]
            assert f"{std / fl:.1f}" == row[4]
            assert std / fl == 1 + n / 128   # the ratio the page states
        elif row[0] == "context":
            assert T.max_context(32, 128, 20 * GIB, flash=(row[1] == "flash")) == int(row[2])


def test_page3_models():
    g = {k: float(v[0]) for k, v in _kv("page3_traffic.txt").items()}
    d = int(g["d"])
    assert 4096 * 4096 == g["entries_4096"]
    assert T.naive_score_bytes(4096, 4096) == g["score_mib_4096"] * MIB
    assert 300e12 / 2e12 == g["balance_flop_per_byte"]
    assert 5 / 4 == g["softmax_intensity"]
    assert T.p3_block_cols(int(g["sram_numbers"]), d) == g["block_cols"]
    assert 4096 // int(g["block_cols"]) == g["passes_4096"]
    assert round(T.p3_standard_bytes(4096, d) / 1e5) / 10 == g["standard_mb_4096"]
    assert round(T.p3_standard_bytes(8192, d) / 1e5) / 10 == g["standard_mb_8192"]
    assert round(T.p3_tiled_bytes(4096, d, 65536) / 1e5) / 10 == g["tiled_mb_4096"]
    assert round(T.p3_tiled_bytes(8192, d, 65536) / 1e5) / 10 == g["tiled_mb_8192"]
    assert round(T.p3_standard_bytes(4096, d) / T.p3_tiled_bytes(4096, d, 65536), 1) == g["ratio_4096"]
    assert round(T.seconds(T.forward_flops(4096, 4096, d), 300e12) * 1e7) / 10 == g["matmul_us_4096"]
    assert (round(T.seconds(T.p3_standard_bytes(4096, d), 2e12) * 1e7) / 10
            == g["standard_traffic_us_4096"])
    assert (round(T.seconds(T.p3_tiled_bytes(4096, d, 65536), 2e12) * 1e7) / 10
            == g["tiled_memory_us_4096"])
    # d = 64 is forced: d = 128 does not reproduce the tiled figure
    assert round(T.p3_tiled_bytes(4096, 128, 65536) / 1e5) / 10 != g["tiled_mb_4096"]


def test_counter_scales_with_heads_and_batch():
    # "Does the traffic grow with the number of heads?" (page 3): x heads x batch
    one = T.compulsory_bytes(4096, 4096, 128)
    assert T.compulsory_bytes(4096, 4096, 128, h_q=32, batch=3) == 96 * one
    # GQA: K and V once per KV head
    assert T.compulsory_bytes(1, 8192, 128, h_q=32, h_kv=8, batch=16) == \
        16 * 2 * 128 * (2 * 32 * 1 + 2 * 8 * 8192)
    assert T.forward_flops(4096, 4096, 128, causal=True, h_q=32) == 32 * 2 * 4096 * 4096 * 128
    assert math.isclose(T.forward_flops(8192, 8192, 128), 34359738368.0)
