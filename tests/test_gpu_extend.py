"""GPU parity of the chunked extend on the expanded path (mla_extend_chunked: expansion
GEMM + flash attention per chunk, chunks merged by LSE) against the oracle's
extend_chunked_expanded, through the C ABI, with the parity bounds of the decode."""
import numpy as np
import pytest
import torch

import oracle
from mla_absorbed_decode_gb300 import workloads as W

from _harness import compare, expanded_score_allowance, to_np

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
