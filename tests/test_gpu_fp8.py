"""GPU parity of the FP8-cache decode (mla_decode_fp8) against the oracle's decode over
the dequantized cache, through the C ABI.  The cases mirror the bf16 decode's: several
pages, ragged tails, forced split-KV, s_q = 2 with causal masking, more rows than one
CTA pair, empty requests, poisoned memory, rescaling, and the full-size V3 shape sampled.
"""
import numpy as np
import pytest
import torch

from mla_absorbed_decode_gb300 import workloads as W

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


def _case(B, s_q, H, seqlens, causal=False, outlier_p=0.0, seed=0, kv_scale=1.0 / 64.0):
    w = W.Workload("fp8_case", B=B, s_q=s_q, H=H, causal=causal, fixed_seqlens=tuple(seqlens),
                   outlier_p=outlier_p, outlier_scale=8.0, kv_fp8=True, kv_scale=kv_scale)
    return make(w, seed=seed)


def test_fp8_smallest():
    inp = _case(1, 1, 16, [1], seed=1)
    ref_out, ref_lse, _ = oracle_decode(inp)
    out, lse, _, _ = run_library(inp)
    compare(out, lse, ref_out, ref_lse, what="fp8 one token")


@pytest.mark.parametrize("H,seqlens", [(16, [63, 64, 65]), (128, [64 * 5 + 7, 1000]), (64, [130, 2, 511]),
                                        (128, [4096])])
def test_fp8_unsplit_and_split(H, seqlens):
    inp = _case(len(seqlens), 1, H, seqlens, seed=H + len(seqlens))
    ref_out, ref_lse, _ = oracle_decode(inp)
    for parts in (None, 1, 2, 5, 13):
        out, lse, _, P = run_library(inp, parts=parts)
        compare(out, lse, ref_out, ref_lse, what=f"fp8 H={H} seqlens={seqlens} parts={P}")


@pytest.mark.parametrize("kv_scale", [0.0123, 0.5])
def test_fp8_scale(kv_scale):
    # a scale that is not a power of two, and one that makes the values (and scores) large
    inp = _case(2, 1, 128, [300, 777], seed=2, kv_scale=kv_scale)
    ref_out, ref_lse, ref_abs = oracle_decode(inp)
    out, lse, _, _ = run_library(inp, parts=3)
    compare(out, lse, ref_out, ref_lse, ref_abs=ref_abs, what=f"fp8 kv_scale={kv_scale}")


@pytest.mark.parametrize("s_q,H", [(2, 128), (2, 16), (3, 128), (4, 128), (3, 40), (2, 20), (3, 127)])
def test_fp8_causal_query_rows(s_q, H):
    seqlens = [2, 65, 300, 1025]
    inp = _case(len(seqlens), s_q, H, seqlens, causal=True, seed=s_q * 100 + H)
    ref_out, ref_lse, _ = oracle_decode(inp)
    for parts in (None, 3):
        out, lse, _, P = run_library(inp, parts=parts)
        compare(out, lse, ref_out, ref_lse, what=f"fp8 s_q={s_q} H={H} parts={P}")


def test_fp8_empty_and_degenerate_requests():
    inp = _case(3, 2, 16, [0, 1, 3], causal=True, seed=3)
    ref_out, ref_lse, _ = oracle_decode(inp)
    out, lse, _, _ = run_library(inp, parts=2)
    compare(out, lse, ref_out, ref_lse, what="fp8 degenerate")
    assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))


def test_fp8_poison_never_reaches_the_result():
    seqlens = [100, 129, 64]
    inp = _case(3, 1, 128, seqlens, seed=11)
    bt = inp["block_table"]
    inp["block_table"] = torch.cat([bt, torch.full((3, 4), -1, dtype=torch.int32)], dim=1)
    assert int((inp["kv_cache"] == 0x7F).sum()) > 0          # NaN codes fill the unused slots
    ref_out, ref_lse, _ = oracle_decode(inp)
    out, lse, _, _ = run_library(inp, parts=4)
    compare(out, lse, ref_out, ref_lse, what="fp8 poison")
    clean = _case(3, 1, 128, seqlens, seed=11)
    kv = clean["kv_cache"]
    kv[kv == 0x7F] = 0
    out2, lse2, _, _ = run_library(clean, parts=4)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


def test_fp8_outlier_rows_and_rescaling():
    # x8 outlier rows make the running maximum jump past the rebase threshold often
    inp = _case(2, 1, 128, [3000, 5000], outlier_p=0.02, seed=5)
    ref_out, ref_lse, ref_abs = oracle_decode(inp)
    for parts in (None, 6):
        out, lse, _, P = run_library(inp, parts=parts)
        compare(out, lse, ref_out, ref_lse, ref_abs=ref_abs, what=f"fp8 outliers parts={P}")


def test_fp8_deterministic():
    inp = _case(2, 1, 128, [700, 3000], seed=9)
    a = run_library(inp, parts=5)
    b = run_library(inp, parts=5)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_fp8_full_size_v3_sampled():
    # the bench's FP8 workload, in its launch configuration, sampled against the oracle
    w = W.FP8
    inp = make(w)
    out, lse, _, _ = run_library(inp)
    sel = sorted({0, w.B - 1, *np.random.default_rng(1).choice(w.B, size=4, replace=False).tolist()})
    ref_out, ref_lse, _ = oracle_decode(inp, sel)
    compare(out[sel], lse[sel], ref_out, ref_lse, what=f"{w.name} sampled {sel}")


def test_fp8_step_chain_and_graph_vs_expanded_definition():
    # DecodeStep over an FP8 cache (absorb with RoPE -> mla_decode_fp8 -> un-absorb), run eagerly
    # and replayed from a CUDA graph, against the expanded (un-absorbed) definition over the
    # dequantized cache
    import oracle
    import mla_absorbed_decode_gb300 as mla
    from _harness import OUT_ABS, to_np
    w = W.small_variant(W.FP8, B=3, seqlen=700)
    inp = make(w)
    B, s_q, H = w.B, w.s_q, w.H
    pos = (inp["seqlens"] - 1).to(torch.int32)
    step = mla.DecodeStep(B, s_q, H, inp["seqlens"].cuda(), w.causal, w.softmax_scale, kv_scale=inp["kv_scale"])
    args = (inp["q_nope"].cuda(), inp["q_pe"].cuda(), inp["w_uk"].cuda(), inp["w_uv"].cuda(),
            inp["kv_cache"].cuda(), inp["block_table"].cuda())
    o = step.run(*args, positions=pos.cuda()).clone()
    assert mla.get_device_status() == 0
    step.capture(*args, positions=pos.cuda())
    o2 = step.replay().clone()
    torch.cuda.synchronize()
    assert mla.get_device_status() == 0
    assert torch.equal(o, o2)
    qp = np.swapaxes(oracle.rope_interleaved(np.swapaxes(to_np(inp["q_pe"]), 0, 1), pos.numpy()), 0, 1)
    kv = oracle.dequantize_e4m3(inp["kv_cache"].numpy(), inp["kv_scale"])
    ref, _ = oracle.decode_expanded(to_np(inp["q_nope"]).reshape(B, s_q, H, 128), qp.reshape(B, s_q, H, 64),
                                    to_np(inp["w_uk"]), to_np(inp["w_uv"]), kv, inp["block_table"].numpy(),
                                    inp["seqlens"].numpy(), w.softmax_scale)
    got = to_np(o.view(B, s_q, H, 128).cpu())
    d = np.abs(got - ref)
    assert d.max() <= OUT_ABS, d.max()
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= 2e-2
