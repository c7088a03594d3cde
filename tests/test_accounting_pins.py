"""The FLOP / byte counters the bench uses, pinned to the numbers the pages print.

Fixtures: tests/golden/flop_counter_mla_paths.json and arithmetic_intensity.json
(each names the page and section its numbers come from).
"""
import json
import os

import pytest

from mla_absorbed_decode_gb300 import accounting as acc

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLD, name), encoding="utf-8") as f:
        return json.load(f)


def test_pair_and_fixed_costs_match_printed_counter():
    p = _load("flop_counter_mla_paths.json")["printed"]
    naive, absorb = acc.pair_flops(128, False), acc.pair_flops(128, True)
    assert f"{naive / 1e3:.0f}" == p["pair_expand_kflops"]
    assert f"{absorb / 1e3:.0f}" == p["pair_absorb_kflops"]
    assert f"{absorb / naive:.1f}" == p["pair_ratio"]
    assert absorb == 278528
    assert f"{acc.fixed_flops(128, False) / 1e6:.1f}" == p["expand_per_key_token_mflops"]
    assert f"{acc.fixed_flops(128, True) / 1e6:.1f}" == p["absorb_per_query_token_mflops"]


def test_path_totals_match_printed_cases():
    p = _load("flop_counter_mla_paths.json")["printed"]
    for case in p["cases"]:
        e, a = acc.path_flops(case["q"], case["k"], 128)
        assert f"{e / 1e9:,.1f}" == case["expand_gflops"], case["what"]
        assert f"{a / 1e9:,.1f}" == case["absorb_gflops"], case["what"]
        assert ("expand" if e < a else "absorb") == case["choice"]


def test_crossover_and_intensity():
    p = _load("flop_counter_mla_paths.json")["printed"]
    assert f"{acc.crossover_new_tokens(128):.0f}" == p["crossover_new_tokens"]
    # decode AI as the counter prints it: per-pair FLOPs over the 1152 cached bytes
    assert f"{acc.pair_flops(128, True) / ((512 + 64) * 2):.0f}" == p["decode_ai_mla_flop_per_byte"]
    assert f"{989e12 / 3.35e12:.0f}" == p["h800_knee_flop_per_byte"]
    # FP8 KV (1 byte per value): about 484 FLOP/B
    assert round(acc.pair_flops(128, True) / 576) == p["fp8_kv_ai_flop_per_byte_approx"]


def test_appendix_a_intensity_and_table():
    p = _load("arithmetic_intensity.json")["printed"]
    for key in ("deepseek_v3", "kimi_k3"):
        c = p[key]
        assert f"{acc.arithmetic_intensity(c['H'], c['d_c'], c['d_s']):.1f}" == c["ai"]
    # without the RoPE part the intensity is exactly 2H in bf16
    assert acc.arithmetic_intensity(128, 512, 0) == p["no_rope_bf16_deepseek"]["ai"]
    t = p["a3_table_per_head_per_pair"]
    # the table counts multiply-adds per head
    assert acc.pair_flops(1, True) // 2 == t["absorb_with_rope"]
    assert acc.pair_flops(1, False) // 2 == t["expand_with_rope"]
    assert acc.fixed_flops(1, False) // 2 == t["prep"]
    assert f"{t['absorb_with_rope'] / t['expand_with_rope']:.1f}" == t["ratio_with_rope"]
    assert (acc.pair_flops(1, True) - acc.pair_flops(1, False)) // 2 == t["difference"]
    for name, bp in p["balance_points"].items():
        assert round(bp["flops"] / bp["bw"]) == bp["knee"], name


def test_decode_work_counts():
    # one request, one query, L tokens: pairs = L
    f, b = acc.decode_work([4096], 1, 128, False)
    assert f == 4096 * 278528
    rows = 128
    assert b == 4096 * 1152 + rows * 1152 + rows * 1024 + rows * 4 + 64 * 4 + 4
    # causal s_q = 2: pairs = 2L - 1 (the counter's q*k - q(q-1)/2)
    f2, _ = acc.decode_work([8192], 2, 128, True)
    assert f2 == acc.causal_pairs(2, 8192) * 278528 == (2 * 8192 - 1) * 278528
    # empty request does no work and reads no cache
    f0, b0 = acc.decode_work([0], 1, 16, False)
    assert f0 == 0 and b0 == 16 * (1152 + 1024 + 4) + 4
    # FP8 cache: 576 bytes per cached token, the rest unchanged; per-pair FLOPs over the
    # cached bytes is the printed ~484 FLOP/B of exercise 2
    f8, b8 = acc.decode_work([4096], 1, 128, False, kv_value_bytes=acc.FP8)
    assert f8 == f and b8 == b - 4096 * 576
    p = _load("flop_counter_mla_paths.json")["printed"]
    assert round(f8 / (4096 * 576)) == p["fp8_kv_ai_flop_per_byte_approx"]


@pytest.mark.parametrize("absorb", [True, False])
def test_bmm_work(absorb):
    f, b = acc.bmm_work(64, 128, absorb)
    assert f == 2 * 64 * 128 * 128 * 512
    assert b > 128 * 128 * 512 * 2


def test_sparse_decode_work_counts():
    # every token of a request listed once: the same pairs and cache bytes as the dense
    # decode; on top, 4 bytes per list entry and the list length
    L = 4096
    full = list(range(L))
    f, b = acc.sparse_decode_work([L], [L], 1, 128, False, indices=[full])
    fd, bd = acc.decode_work([L], 1, 128, False)
    assert f == fd
    assert b == bd + L * 4 + 4
    # 2048 of 16384 tokens: pairs = k per query, bytes = k cached rows + q/out/lse + lists
    f, b = acc.sparse_decode_work([16384], [2048], 1, 128, False)
    assert f == 2048 * 278528
    assert b == 2048 * 1152 + 128 * (1152 + 1024 + 4) + 2048 * 4 + min(2048, 256) * 4 + 8
    # causal, s_q = 2, seqlen 10: listed positions 3, 8, 9; query 0 sees t <= 8, query 1 t <= 9
    f, _ = acc.sparse_decode_work([10], [3], 2, 16, True, indices=[[3, 8, 9]])
    assert f == (2 + 3) * 16 * 2176
    # over an FP8 cache a listed token costs 576 bytes, the rest unchanged
    f8, b8 = acc.sparse_decode_work([16384], [2048], 1, 128, False, kv_value_bytes=acc.FP8)
    assert f8 == 2048 * 278528 and b8 == 2048 * 576 + 128 * (1152 + 1024 + 4) + 2048 * 4 + min(2048, 256) * 4 + 8
