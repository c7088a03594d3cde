"""GPU parity of the absorbed decode path against the CPU oracle, through the C ABI.

Small cases (the oracle finishes in seconds) cover several pages, ragged tails,
forced split-KV, s_q = 2 with causal masking, empty requests and poisoned
memory.  The full-size workloads run in the launch configuration the bench
times and are compared on sampled requests.
"""
import math

import numpy as np
import pytest
import torch

from mla_absorbed_decode_gb300 import workloads as W
from oracle.schedule import check_schedule, schedule_reference

from _harness import compare, make, oracle_decode, run_library

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_absorbed_decode_gb300 import build_lib
    build_lib.build()
    import mla_absorbed_decode_gb300 as mla
    mla.lib()
    yield


def _case(B, s_q, H, seqlens, causal=False, outlier_p=0.0, seed=0):
    w = W.Workload("case", B=B, s_q=s_q, H=H, causal=causal, fixed_seqlens=tuple(seqlens),
                   outlier_p=outlier_p, outlier_scale=8.0)
    return make(w, seed=seed)


def test_tiny_workload():
    inp = make(W.TINY)
    out, lse, _, _ = run_library(inp)
    ref_out, ref_lse, ref_abs = oracle_decode(inp)
    compare(out, lse, ref_out, ref_lse, what="tiny")


def test_schedule_bit_exact():
    import mla_absorbed_decode_gb300 as mla
    fixed, hbm, split_cost = mla.schedule_params()
    rng = np.random.default_rng(0)
    cases = [[4096] * 64, [131072] * 4, [256, 300], [0, 5, 0, 700, 64, 65, 0]]
    for _ in range(12):
        B = int(rng.integers(1, 200))
        cases.append([int(x) for x in rng.choice([0, int(rng.integers(1, 64)), int(rng.integers(1, 9000))], size=B)])
    # more requests than the schedule kernel has threads: several requests per thread
    for B in (513, 3000, 16384):
        cases.append([int(x) for x in rng.integers(0, 9000, size=B)])
    for seqlens in cases:
        for P in ((1, 3, 17, 38, 64, 74, 76, 148) if len(seqlens) < 512 else (5, 76, 148)):
            sl = torch.tensor(seqlens, dtype=torch.int32, device="cuda")
            meta = mla.decode_metadata(sl, 1, 128, False, P).cpu().numpy()
            ref_meta, ref_ns = schedule_reference(seqlens, P, fixed, hbm, split_cost)
            got = [tuple(int(v) for v in meta[8 * p: 8 * p + 5]) for p in range(P)]
            assert got == ref_meta, (seqlens[:8], P)
            assert list(meta[8 * P:]) == ref_ns
            check_schedule(got, ref_ns, seqlens)


@pytest.mark.parametrize("H,seqlens", [(16, [1]), (16, [63, 64, 65]), (128, [64 * 5 + 7, 1000]), (64, [130, 2, 511]),
                                        (128, [4096])])
def test_small_unsplit_and_split(H, seqlens):
    inp = _case(len(seqlens), 1, H, seqlens, seed=H + len(seqlens))
    ref_out, ref_lse, ref_abs = oracle_decode(inp)
    for parts in (None, 1, 2, 5, 13):
        out, lse, meta, P = run_library(inp, parts=parts)
        compare(out, lse, ref_out, ref_lse, what=f"H={H} seqlens={seqlens} parts={P}")


@pytest.mark.parametrize("H", [16, 64, 128])
def test_mtp_causal_two_queries(H):
    seqlens = [2, 65, 300, 1025]
    inp = _case(len(seqlens), 2, H, seqlens, causal=True, seed=7)
    ref_out, ref_lse, ref_abs = oracle_decode(inp)
    for parts in (None, 3):
        out, lse, _, P = run_library(inp, parts=parts)
        compare(out, lse, ref_out, ref_lse, what=f"s_q=2 H={H} parts={P}")


@pytest.mark.parametrize("s_q,H", [(3, 128), (4, 128), (2, 80), (3, 40)])
def test_more_query_rows_than_one_pair(s_q, H):
    # s_q * H rows beyond 128 go to further CTA pairs of the same cluster (up to four,
    # a cluster of eight CTAs); the last pair may be partly filled
    seqlens = [5, 200, 1100]
    inp = _case(len(seqlens), s_q, H, seqlens, causal=True, seed=s_q * 1000 + H)
    ref_out, ref_lse, ref_abs = oracle_decode(inp)
    for parts in (None, 4):
        out, lse, _, P = run_library(inp, parts=parts)
        compare(out, lse, ref_out, ref_lse, what=f"s_q={s_q} H={H} parts={P}")


@pytest.mark.parametrize("s_q,H", [(1, 1), (1, 20), (1, 127), (2, 20), (2, 100), (3, 127)])
def test_head_counts_off_the_tile(s_q, H):
    # s_q * H rows that leave part of a 128-row block unused, and (causal) rows whose
    # query position i = row // H changes inside a warp
    seqlens = [3, 64, 190, 700]
    inp = _case(len(seqlens), s_q, H, seqlens, causal=s_q > 1, seed=s_q * 7 + H)
    ref_out, ref_lse, ref_abs = oracle_decode(inp)
    for parts in (None, 1, 5):
        out, lse, _, P = run_library(inp, parts=parts)
        compare(out, lse, ref_out, ref_lse, what=f"s_q={s_q} H={H} parts={P}")


def test_largest_batch():
    # the schedule's maximum batch (16384 requests), short contexts, sampled against the oracle
    B = 16384
    seqlens = np.random.default_rng(4).integers(1, 200, size=B).tolist()
    inp = _case(B, 1, 16, seqlens, seed=4)
    out, lse, _, _ = run_library(inp)
    sel = [0, 1, 777, 8191, B - 2, B - 1]
    # the oracle on the sampled requests only: their pages gathered into a small cache
    bt = inp["block_table"][sel]
    pages = sorted({int(x) for x in bt.flatten().tolist() if x >= 0})
    remap = {pg: i for i, pg in enumerate(pages)}
    sub = dict(inp, q=inp["q"][sel], seqlens=inp["seqlens"][sel], kv_cache=inp["kv_cache"][pages],
               block_table=bt.clone().apply_(lambda x: remap.get(x, -1)))
    ref_out, ref_lse, ref_abs = oracle_decode(sub)
    compare(out[sel], lse[sel], ref_out, ref_lse, what="B=16384")


def test_empty_and_degenerate_requests():
    # an empty request, one token, and s_q > seqlen under causal masking
    inp = _case(3, 2, 16, [0, 1, 3], causal=True, seed=3)
    ref_out, ref_lse, ref_abs = oracle_decode(inp)
    out, lse, _, _ = run_library(inp, parts=2)
    compare(out, lse, ref_out, ref_lse, what="degenerate")
    assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))


def test_poison_never_reaches_the_result():
    seqlens = [100, 129, 64]
    inp = _case(3, 1, 128, seqlens, seed=11)
    # NaN already fills unused slots and pages; add garbage block-table entries past the end
    bt = inp["block_table"]
    inp["block_table"] = torch.cat([bt, torch.full((3, 4), -1, dtype=torch.int32)], dim=1)
    ref_out, ref_lse, ref_abs = oracle_decode(inp)
    out, lse, _, _ = run_library(inp, parts=4)
    compare(out, lse, ref_out, ref_lse, what="poison")
    # the same inputs without poison give the same bits
    clean = _case(3, 1, 128, seqlens, seed=11)
    clean["kv_cache"] = torch.nan_to_num(clean["kv_cache"], nan=0.0)
    out2, lse2, _, _ = run_library(clean, parts=4)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


def test_outlier_rows_and_rescaling():
    # x8 outlier rows make the running maximum jump, which exercises the O rescale path
    inp = _case(2, 1, 128, [3000, 5000], outlier_p=0.02, seed=5)
    ref_out, ref_lse, ref_abs = oracle_decode(inp)
    for parts in (None, 6):
        out, lse, _, P = run_library(inp, parts=parts)
        compare(out, lse, ref_out, ref_lse, ref_abs=ref_abs, what=f"outliers parts={P}")


def test_deterministic():
    inp = _case(2, 1, 128, [700, 3000], seed=9)
    a = run_library(inp, parts=5)
    b = run_library(inp, parts=5)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


# ------------------------------------------------------------- full-size workloads --

def _sample(B, k=4):
    return sorted({0, B - 1, *np.random.default_rng(1).choice(B, size=min(k, B), replace=False).tolist()})


@pytest.mark.parametrize("w", [W.V3, W.RAGGED, W.MTP, W.LONG], ids=lambda w: w.name)
def test_full_size_workload_sampled(w):
    inp = make(w)
    out, lse, _, P = run_library(inp)
    sel = _sample(w.B) if w.B > 4 else list(range(w.B))
    if w.name == W.LONG.name:
        sel = [0, 3]
    ref_out, ref_lse, ref_abs = oracle_decode(inp, sel)
    compare(out[sel], lse[sel], ref_out, ref_lse, ref_abs=ref_abs if w.outlier_p > 0 else None,
            what=f"{w.name} sampled {sel}")


# ------------------------------------------------------------------ mutations --

def _marker_case(seed=13):
    """One 4096-token request whose result hinges on eight marker tokens.  Every head's
    RoPE query part is set to one vector u (|u|^2 = 64) and the markers' RoPE key part to
    3u, so each marker scores ~14 nats above the random tokens for every head and the
    eight of them carry nearly all the softmax weight; their latent (value) parts stay
    N(0,1) draws, so the output keeps unit scale.  A kernel that drops any marker, or
    reads the wrong page for one, moves the output by ~1/8 of a unit value -- far
    outside the parity bounds -- whereas with random inputs alone a single token's
    weight (~1/4096) would sit inside them."""
    inp = _case(1, 1, 128, [4096], seed=seed)
    g = torch.Generator().manual_seed(seed)
    u = torch.randn(64, generator=g)
    u = u / u.norm() * 8.0
    inp["q"][..., 512:576] = u.to(torch.bfloat16)
    markers = [63, 64, 511, 1000, 2047, 2048, 3333, 4095]       # page ends and starts among them
    bt = inp["block_table"][0]
    for t in markers:
        inp["kv_cache"][bt[t // 64], t % 64, 512:576] = (3.0 * u).to(torch.bfloat16)
    return inp, markers


def test_harness_catches_a_dropped_token_and_a_wrong_page():
    import mla_absorbed_decode_gb300 as mla
    inp, markers = _marker_case()
    ref_out, ref_lse, _ = oracle_decode(inp)
    out, lse, _, _ = run_library(inp, parts=4)                  # split over parts, as the bench runs it
    compare(out, lse, ref_out, ref_lse, what="marker case")
    # mutation 1: the last token (a marker) dropped by the kernel's input
    short = dict(inp)
    short["seqlens"] = inp["seqlens"] - 1
    out1, lse1, _, _ = run_library(short, parts=4)
    with pytest.raises(AssertionError):
        compare(out1, lse1, ref_out, ref_lse, what="dropped token")
    # mutation 2: the page holding marker 1000 replaced by its neighbour page (one page read twice)
    shifted = dict(inp)
    bt = inp["block_table"].clone()
    bt[0, 1000 // 64] = bt[0, 1000 // 64 + 1]
    shifted["block_table"] = bt
    out2, lse2, _, _ = run_library(shifted, parts=4)
    with pytest.raises(AssertionError):
        compare(out2, lse2, ref_out, ref_lse, what="wrong page")
    assert mla.get_device_status() == 0
