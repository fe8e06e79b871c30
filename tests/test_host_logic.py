"""Host-side logic against the worked examples the FP32 FlashAttention-2 blog
prints (fixture tests/golden/fa2_v2_blog_worked_examples.json, each entry
citing its section)."""
import json
import os

import pytest

import online_softmax_attention_attn_gb300 as pkg
from online_softmax_attention_attn_gb300 import metrics

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                   "fa2_v2_blog_worked_examples.json")))


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(pkg.LIB_PATH):
        from online_softmax_attention_attn_gb300 import _build
        _build.build()
    return pkg.lib()


def test_grid_of_q_blocks(L):
    g = GOLD["grid"]
    n_qblocks = -(-g["N"] // g["Br"])
    assert n_qblocks == g["grid_x"]
    assert g["B"] * g["H"] == g["grid_y"]
    assert n_qblocks * g["B"] * g["H"] == g["ctas"]


def test_nvec(L):
    g = GOLD["nvec"]
    assert g["Bc"] * g["D"] // 4 == g["nvec"]


def test_causal_block_skipping_worked_example(L):
    g = GOLD["causal_skip"]
    row_begin = g["q_block"] * g["Br"]
    assert (row_begin, row_begin + g["Br"]) == (g["row_begin"], g["row_end"])
    tiles = pkg.attn_kv_tiles(g["N"], g["Br"], g["Bc"], True, g["q_block"])
    assert tiles == g["kv_blocks_processed"]
    total = pkg.attn_kv_tiles(g["N"], g["Br"], g["Bc"], False, g["q_block"])
    assert total - tiles == g["kv_blocks_skipped"]
    assert tiles * g["Bc"] == g["kv_limit"]


def test_kv_tiles_edges(L):
    assert pkg.attn_kv_tiles(256, 128, 128, True, 0) == 1
    assert pkg.attn_kv_tiles(256, 128, 128, True, 1) == 2
    assert pkg.attn_kv_tiles(300, 128, 128, True, 2) == 3   # ragged last block
    assert pkg.attn_kv_tiles(300, 128, 64, False, 0) == 5
    assert pkg.attn_kv_tiles(1, 128, 128, True, 0) == 1
    assert pkg.attn_kv_tiles(300, 128, 128, True, 3) == -1  # past the end


def test_blog_shared_memory_budget():
    g = GOLD["smem_bytes"]
    Br, Bc, D = g["Br"], g["Bc"], g["D"]
    bytes_ = (2 * Bc * D + 2 * Bc * D + 2 * Br * (D + 1)) * 4
    assert bytes_ == g["bytes"]
    assert round(bytes_ / 1024) == g["about_kib"]


def test_flop_convention_reproduces_the_timing_table():
    t = GOLD["timing_table"]
    for row in t["rows"]:
        f = metrics.mha_flops(t["B"], t["H"], t["N"], t["D"], row["causal"])
        tflops = f / (row["ms"] * 1e-3) / 1e12
        # the page prints times to 2-5 significant digits
        assert abs(tflops - row["tflops"]) / row["tflops"] < 0.025, (row, tflops)


def test_mla_bytes_of_the_uniform_decode_workload():
    # batch 64, Hq 128, seq 4096, identity table of 64 pages per sequence
    b = metrics.mla_bytes([4096] * 64, max_blocks=64)
    assert b == 301989888 + 9437184 + 8388608 + 32768 + 16384 + 256
