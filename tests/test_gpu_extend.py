"""GPU parity of the chunked extend on the expanded path (mla_extend_chunked: expansion
GEMM + flash attention per chunk, chunks merged by LSE) against the oracle's
extend_chunked_expanded, through the C ABI, with the parity bounds of the decode."""
import numpy as np
import pytest
import torch

import oracle
from mla_absorbed_decode_gb300 import workloads as W

from _harness import compare, expanded_output_allowance, expanded_score_allowance, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_absorbed_decode_gb300 import build_lib
    build_lib.build()
    yield


def _case(T, seqlen, H, seed):
    w = W.Workload("extend", B=1, s_q=T, H=H, fixed_seqlens=(seqlen,), with_projections=True)
    return W.make_inputs(w, seed=seed)   # unused pages and the last page's tail hold NaN


def _run(inp, seqlen, chunk):
    import mla_absorbed_decode_gb300 as mla
    out, lse = mla.extend_chunked(inp["q_nope"].cuda(), inp["q_pe"].cuda(), inp["w_uk"].cuda(), inp["w_uv"].cuda(),
                                  inp["kv_cache"].cuda(), inp["block_table"][0].contiguous().cuda(), seqlen,
                                  inp["softmax_scale"], chunk_tokens=chunk)
    assert mla.get_device_status() == 0
    return out.cpu(), lse.cpu()


def _ref(inp, seqlen, chunk):
    return oracle.extend_chunked_expanded(to_np(inp["q_nope"]), to_np(inp["q_pe"]), to_np(inp["w_uk"]),
                                          to_np(inp["w_uv"]), inp["kv_cache"].float().numpy(),
                                          inp["block_table"][0].numpy(), seqlen, inp["softmax_scale"], chunk)


def _allowance(inp, seqlen):
    """The lse allowance for the bf16 expanded keys (expanded_score_allowance)."""
    rows = oracle.gather_request(inp["kv_cache"].float().numpy(), inp["block_table"][0].numpy(), seqlen)
    k_nope, _, _ = oracle.expand_chunk(rows, to_np(inp["w_uk"]), to_np(inp["w_uv"]))
    T = inp["q_nope"].shape[0]
    return expanded_score_allowance(to_np(inp["q_nope"]), k_nope, inp["softmax_scale"], np.arange(seqlen - T, seqlen))


@pytest.mark.parametrize("T,seqlen,H,chunks", [
    (5, 300, 4, (64, 128, 320)),       # many chunks, one chunk; a ragged last page
    (130, 700, 2, (256,)),             # two query tiles, causal across them
    (64, 64, 8, (64,)),                # a prefill without a prefix (T = seqlen)
    (3, 256, 128, (128,)),             # all 128 heads
    (37, 2100, 16, (1024, 2048)),      # a longer prefix, a chunk boundary inside a query tile's view
    (300, 300, 2, (64, 128)),          # a prefill of three query tiles: the first sees none of the later chunks
])
def test_extend_chunked_matches_the_oracle(T, seqlen, H, chunks):
    inp = _case(T, seqlen, H, seed=T + seqlen + H)
    extra = _allowance(inp, seqlen)
    ref_o, ref_l = None, None
    for chunk in chunks:
        out, lse = _run(inp, seqlen, chunk)
        if ref_o is None:   # the merged result does not depend on the chunking (an oracle pin)
            ref_o, ref_l = _ref(inp, seqlen, chunk)
        compare(out, lse, ref_o, ref_l, what=f"extend T={T} L={seqlen} H={H} chunk={chunk}", lse_extra=extra)


def test_extend_equals_the_absorbed_chain_on_the_gpu():
    # the pages' claim, on the GPU: W_UK absorbed, attention over the latent, W_UV last
    import mla_absorbed_decode_gb300 as mla
    T, seqlen, H = 4, 900, 64
    inp = _case(T, seqlen, H, seed=77)
    out_x, lse_x = _run(inp, seqlen, 256)
    q = torch.empty((1, T, H, 576), dtype=torch.bfloat16, device="cuda")
    mla.absorb_q(inp["q_nope"].cuda(), inp["w_uk"].cuda(), q.view(T, H, 576), q_pe=inp["q_pe"].cuda())
    sl = inp["seqlens"].cuda()
    P = mla.num_sm_parts(T, H)
    meta = mla.decode_metadata(sl, T, H, True, P)
    lat, lse_a = mla.decode(q, inp["kv_cache"].cuda(), inp["block_table"].cuda(), sl, inp["softmax_scale"], True, meta, P)
    o_a = mla.unabsorb_o(lat.view(T, H, 512), inp["w_uv"].cuda())
    assert mla.get_device_status() == 0
    compare(out_x, lse_x, to_np(o_a.cpu()), to_np(lse_a[0].cpu()), what="expanded vs absorbed on the GPU",
            lse_extra=_allowance(inp, seqlen))


def test_extend_reports_a_bad_block_table_entry():
    import mla_absorbed_decode_gb300 as mla
    T, seqlen, H = 4, 200, 4
    inp = _case(T, seqlen, H, seed=5)
    row = inp["block_table"][0].clone()
    row[1] = inp["kv_cache"].shape[0] + 3
    mla.extend_chunked(inp["q_nope"].cuda(), inp["q_pe"].cuda(), inp["w_uk"].cuda(), inp["w_uv"].cuda(),
                       inp["kv_cache"].cuda(), row.cuda(), seqlen, inp["softmax_scale"], chunk_tokens=64)
    assert mla.get_device_status() == 6      # MLA_ERR_DEVICE_BOUNDS
    assert mla.get_device_status() == 0


def _rebases_by_warpgroup(s_log2, L, T, chunk):
    """The attention kernel's rebase rule replayed on exact scores: per chunk, 64-key tiles
    in order; a row's reference maximum moves when a tile's maximum exceeds it by more than
    2^8; tile k of a chunk is processed by softmax warpgroup k % 2.  Counts the moves after
    each chunk's first two tiles, per warpgroup."""
    qpos = np.arange(L - T, L)
    late = [0, 0]
    for c0 in range(0, L, chunk):
        c1 = min(L, c0 + chunk)
        ref = np.full(s_log2.shape[:2], -np.inf)
        for k, t0 in enumerate(range(c0, c1, 64)):
            keys = np.arange(t0, min(c1, t0 + 64))
            vis = keys[None, :] <= qpos[:, None]
            m = np.where(vis[:, None, :], s_log2[:, :, keys], -np.inf).max(axis=2)
            move = m > ref + 8
            if k >= 2:
                late[k % 2] += int(move.sum())
            ref = np.where(move, m, ref)
    return late


def test_extend_rebases_the_reference_maximum_in_both_warpgroups():
    # cache rows scaled x2 .. x8 at planted positions make the row maxima grow past the lazy
    # rebase threshold late in a chunk, on tiles of both parities (both softmax warpgroups:
    # the one whose tile moves the reference rescales O, each rescales its own row sum)
    T, L, H, chunk = 37, 2100, 16, 1024
    inp = _case(T, L, H, seed=11)
    bt = inp["block_table"][0]
    for t, f in {200: 2.0, 520: 4.0, 840: 8.0, 1400: 4.0, 1800: 8.0}.items():
        inp["kv_cache"][bt[t // 64], t % 64] = (inp["kv_cache"][bt[t // 64], t % 64].float() * f).to(torch.bfloat16)
    rows = oracle.gather_request(inp["kv_cache"].float().numpy(), bt.numpy(), L)
    k_nope, k_pe, v = oracle.expand_chunk(rows, to_np(inp["w_uk"]), to_np(inp["w_uv"]))
    qn, qp = to_np(inp["q_nope"]), to_np(inp["q_pe"])
    s = (np.einsum("thd,hnd->thn", qn, k_nope) + np.einsum("thd,nd->thn", qp, k_pe)) * inp["softmax_scale"]
    late = _rebases_by_warpgroup(s * np.log2(np.e), L, T, chunk)
    assert min(late) > 0, late   # the case exercises what it is meant to
    out, lse = _run(inp, L, chunk)
    ref_o, ref_l = _ref(inp, L, chunk)
    # magnitude of each output element (outlier rows are not unit-scale): attention to |v|
    qpos = np.arange(L - T, L)
    ref_abs, _ = oracle.attend_chunk(qn, qp, k_nope, k_pe, np.abs(v), np.arange(L), qpos, inp["softmax_scale"])
    # With x8 rows the scores are large, and rounding the expanded keys to bf16 (the path's
    # definition) moves P by a few percent on rows that a few outlier tokens dominate: the
    # output gets the allowance that follows from the score allowance (a mistake in the
    # rescales would be off by up to a factor of 2^8).
    extra = _allowance(inp, L)
    compare(out, lse, ref_o, ref_l, ref_abs=ref_abs, what="extend with planted outlier rows", lse_extra=extra,
            out_extra=expanded_output_allowance(extra, ref_abs))
