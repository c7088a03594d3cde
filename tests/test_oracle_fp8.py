"""Pins of the oracle's FP8 (E4M3) cache decode, against the format's definition,
a library conversion and the (separately pinned) bf16 decode definition."""
import math

import numpy as np
import pytest
import torch

import oracle
from mla_absorbed_decode_gb300 import workloads as W


def test_e4m3_special_values():
    v = oracle.E4M3_VALUES
    assert v[0x00] == 0.0 and not math.copysign(1.0, v[0x00]) < 0
    assert v[0x80] == 0.0 and math.copysign(1.0, v[0x80]) < 0
    assert v[0x01] == 2.0 ** -9            # smallest subnormal
    assert v[0x07] == 7 * 2.0 ** -9        # largest subnormal
    assert v[0x08] == 2.0 ** -6            # smallest normal
    assert v[0x38] == 1.0 and v[0x3C] == 1.5 and v[0x40] == 2.0
    assert v[0x7E] == 448.0 and v[0xFE] == -448.0
    nan = np.isnan(v)
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    pos = v[0x00:0x7F]
    assert np.all(np.diff(pos) > 0)        # codes 0..126 increase strictly
    assert np.array_equal(v[0x80:0xFF], -v[0x00:0x7F])


def test_e4m3_matches_library_conversion():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    lib = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = oracle.E4M3_VALUES
    same = (lib == mine) | (np.isnan(lib) & np.isnan(mine))
    assert same.all(), np.nonzero(~same)


def test_fp8_decode_equals_bf16_decode_of_the_dequantized_cache():
    # E4M3 values times a power of two are exact in bf16, so the FP8 decode must equal
    # the bf16 decode of the dequantized cache; this pins the gather and the scaling.
    w = W.small_variant(W.FP8, B=3, seqlen=200, H=8)
    d = W.make_inputs(w, seed=1)
    codes = d["kv_cache"].numpy()
    scale = d["kv_scale"]
    assert scale == 2.0 ** -6
    deq = oracle.dequantize_e4m3(codes, scale)
    deq_bf16 = torch.from_numpy(deq).to(torch.bfloat16)
    assert np.array_equal(deq_bf16.to(torch.float64).numpy(), deq, equal_nan=True)
    q, bt, sl = d["q"].float().numpy(), d["block_table"].numpy(), d["seqlens"].numpy()
    o8, l8 = oracle.decode_fp8(q, codes, scale, bt, sl, w.softmax_scale)
    ob, lb = oracle.decode_absorbed(q, deq_bf16.float().numpy(), bt, sl, w.softmax_scale)
    assert np.array_equal(o8, ob) and np.array_equal(l8, lb)
    assert np.isfinite(o8).all()           # the poison codes (NaN) are never read


def test_fp8_single_token_closed_form():
    # one visible token: out = its dequantized value row, lse = its scaled score
    rng = np.random.default_rng(0)
    codes = rng.integers(0, 0x7E, size=(2, 64, 576), dtype=np.uint8)
    scale = 0.0123
    q = rng.standard_normal((1, 1, 4, 576))
    bt = np.array([[1]], dtype=np.int32)
    out, lse = oracle.decode_fp8(q, codes, scale, bt, np.array([1]), softmax_scale=0.07)
    row = oracle.E4M3_VALUES[codes[1, 0]] * scale
    np.testing.assert_allclose(out[0, 0], np.broadcast_to(row[:512], (4, 512)), rtol=1e-15, atol=0)
    np.testing.assert_allclose(lse[0, 0], 0.07 * (q[0, 0] @ row), rtol=1e-12)


@pytest.mark.parametrize("scale", [2.0 ** -6, 0.0123])
def test_fp8_workload_codes_round_the_draws(scale):
    # the generator's codes are the E4M3 rounding of kv / scale: each dequantized value is
    # within half a step of the draw (relative 2^-4 above 2^-6, 2^-10 absolute below)
    w = W.Workload("fp8_probe", B=1, s_q=1, H=1, seqlen=64, kv_fp8=True, kv_scale=scale)
    d = W.make_inputs(w, seed=3, poison=False)
    g = torch.Generator().manual_seed(3)     # the same draws, in make_inputs' order
    pool = math.ceil(1.03 * 1)
    torch.randperm(pool, generator=g)
    torch.randn((1, 1, 1, 576), generator=g)
    draws = (torch.randn((pool, 64, 576), generator=g) / scale).double().numpy()
    codes = d["kv_cache"].numpy()
    x = oracle.E4M3_VALUES[codes]
    assert np.isfinite(x).all() and np.abs(x).max() <= 448.0
    err = np.abs(x - np.clip(draws, -448, 448))
    bound = np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10)
    assert np.all(err <= bound * (1 + 1e-12))


def test_fp8_sparse_decode_equals_bf16_sparse_of_the_dequantized_cache():
    # the sparse (top-k) decode over an FP8 cache: the bf16 sparse decode of the dequantized
    # cache, exactly (E4M3 values times 2^-6 are bf16 numbers)
    w = W.Workload("fp8_sparse_probe", B=2, s_q=2, H=4, seqlen=300, topk=100, causal=True, kv_fp8=True)
    d = W.make_inputs(w, seed=4)
    codes, scale = d["kv_cache"].numpy(), d["kv_scale"]
    deq = torch.from_numpy(oracle.dequantize_e4m3(codes, scale)).to(torch.bfloat16).float().numpy()
    q, bt, sl = d["q"].float().numpy(), d["block_table"].numpy(), d["seqlens"].numpy()
    idx, kl = d["indices"].numpy(), d["topk_lens"].numpy()
    o8, l8 = oracle.decode_sparse(q, codes, bt, sl, idx, kl, w.softmax_scale, causal=True, kv_scale=scale)
    ob, lb = oracle.decode_sparse(q, deq, bt, sl, idx, kl, w.softmax_scale, causal=True)
    assert np.array_equal(o8, ob) and np.array_equal(l8, lb)
    assert np.isfinite(o8).all()
