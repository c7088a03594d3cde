"""Host logic of bench.py that needs no GPU: the committed DRAM traffic of the decode
kernel and the source digest that decides whether bench.py may report it."""
import json
import os

import pytest

import bench
from mla_absorbed_decode_gb300 import accounting as acc
from mla_absorbed_decode_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TRAFFIC = os.path.join(ROOT, "profiles", "decode_traffic.json")
DECODE_WORKLOADS = ("deepseek_v3_b64_h128_l4096", "fp8_deepseek_v3_b64_h128_l4096",
                    "sparse_b64_h128_l16384_top2048", "sparse_fp8_b64_h128_l16384_top2048")


def _entries():
    with open(TRAFFIC) as f:
        return json.load(f)


def _algorithmic_bytes(name):
    """Bytes one decode launch must move at the workload's full size (every request
    has the same length here, so no inputs need to be drawn)."""
    w = W.BY_NAME[name]
    assert w.seqlen > 0 and not w.ragged_max
    lens = [w.seqlen] * w.B
    kvb = acc.FP8 if w.kv_fp8 else acc.BF16
    if w.topk:
        return acc.sparse_decode_work(lens, [min(w.topk, w.seqlen)] * w.B, w.s_q, w.H, w.causal,
                                      kv_value_bytes=kvb)[1]
    return acc.decode_work(lens, w.s_q, w.H, w.causal, kv_value_bytes=kvb)[1]


def test_digest_covers_existing_sources():
    for rel in bench.DECODE_KERNEL_SOURCES:
        assert os.path.exists(os.path.join(ROOT, rel)), rel
    d = bench._source_digest()
    assert len(d) == 16 and int(d, 16) >= 0


@pytest.mark.parametrize("name", DECODE_WORKLOADS)
def test_traffic_entry_is_the_scaled_capture(name):
    e = _entries()[name]
    assert e["dram_bytes_per_launch"] == int(e["captured_bytes"] * e["scale"])
    assert e["scale"] == W.BY_NAME[name].B / 32   # captured at B=32, every term scales with B


@pytest.mark.parametrize("name", DECODE_WORKLOADS)
def test_traffic_is_close_to_the_algorithmic_bytes(name):
    """Each cached row leaves HBM once: the captured DRAM bytes stay within a few percent of
    the algorithmic bytes.  They may fall a little below (part of the output writes is still
    in L2 when the launch ends), and a wasted re-read of the cache would push them well above."""
    got = _entries()[name]["dram_bytes_per_launch"]
    want = _algorithmic_bytes(name)
    assert 0.90 * want <= got <= 1.06 * want, (got, want)


def test_traffic_is_reported_only_for_the_captured_source(monkeypatch):
    name = DECODE_WORKLOADS[0]
    e = _entries()[name]
    monkeypatch.setattr(bench, "_source_digest", lambda: e["source_digest"])
    assert bench._traffic_per_launch(name) == e["dram_bytes_per_launch"]
    monkeypatch.setattr(bench, "_source_digest", lambda: "0" * 16)
    assert bench._traffic_per_launch(name) is None
    assert bench._traffic_per_launch("no_such_workload") is None
