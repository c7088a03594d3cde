"""GPU parity of the sparse (top-k) decode against the oracle's decode_sparse, and
against the dense kernel when every token is listed in order (same rows, same
order: the same bits)."""
import numpy as np
import pytest
import torch

import oracle
from mla_absorbed_decode_gb300 import workloads as W

from _harness import compare, make, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_absorbed_decode_gb300 import build_lib
    build_lib.build()
    yield


def _case(B, s_q, H, seqlens, causal=False, seed=0):
    w = W.Workload("sparse_case", B=B, s_q=s_q, H=H, causal=causal, fixed_seqlens=tuple(seqlens))
    return make(w, seed=seed)


def _lists(seqlens, ks, seed, stride=None):
    rng = np.random.default_rng(seed)
    stride = stride or max(max(ks), 1)
    idx = np.full((len(seqlens), stride), -1, dtype=np.int32)
    for b, (L, k) in enumerate(zip(seqlens, ks)):
        if k:
            idx[b, :k] = np.sort(rng.choice(L, size=k, replace=False))
    return torch.from_numpy(idx), torch.tensor(ks, dtype=torch.int32)


def _run(inp, idx, kl, parts=None):
    import mla_absorbed_decode_gb300 as mla
    q, kv, bt, sl = (inp[k].cuda() for k in ("q", "kv_cache", "block_table", "seqlens"))
    B, s_q, H, _ = q.shape
    P = parts or mla.num_sm_parts(s_q, H)
    meta = mla.decode_metadata(kl.cuda(), s_q, H, inp["causal"], P)
    out, lse = mla.decode_sparse(q, kv, bt, sl, idx.cuda(), kl.cuda(), inp["softmax_scale"], inp["causal"], meta, P)
    assert mla.get_device_status() == 0
    return out.cpu(), lse.cpu()


def _ref(inp, idx, kl):
    return oracle.decode_sparse(to_np(inp["q"]), inp["kv_cache"].float().numpy(), inp["block_table"].numpy(),
                                inp["seqlens"].numpy(), idx.numpy(), kl.numpy(), inp["softmax_scale"],
                                causal=inp["causal"])


@pytest.mark.parametrize("H,s_q,causal", [(16, 1, False), (128, 1, False), (128, 2, True), (64, 2, False),
                                           (20, 2, True), (127, 1, False)])
def test_sparse_small(H, s_q, causal):
    seqlens = [5000, 130, 64, 3000]
    ks = [2048, 130, 1, 777]   # top-k, everything, a single token, ragged
    inp = _case(len(seqlens), s_q, H, seqlens, causal=causal, seed=H + s_q)
    idx, kl = _lists(seqlens, ks, seed=H)
    ref_out, ref_lse = _ref(inp, idx, kl)
    for parts in (None, 3):
        out, lse = _run(inp, idx, kl, parts)
        compare(out, lse, ref_out, ref_lse, what=f"sparse H={H} s_q={s_q} parts={parts}")


def test_sparse_empty_list_and_unsorted_order():
    seqlens = [300, 900]
    inp = _case(2, 1, 64, seqlens, seed=5)
    idx, kl = _lists(seqlens, [0, 500], seed=5)
    idx[1, :500] = idx[1, :500][torch.randperm(500, generator=torch.Generator().manual_seed(1))]
    out, lse = _run(inp, idx, kl)
    ref_out, ref_lse = _ref(inp, idx, kl)
    compare(out, lse, ref_out, ref_lse, what="sparse empty/unsorted")
    assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))


def test_every_token_listed_matches_the_dense_kernel_bit_for_bit():
    import mla_absorbed_decode_gb300 as mla
    seqlens = [1000, 64, 4097]
    inp = _case(3, 1, 128, seqlens, seed=9)
    stride = max(seqlens)
    idx = torch.full((3, stride), -1, dtype=torch.int32)
    for b, L in enumerate(seqlens):
        idx[b, :L] = torch.arange(L, dtype=torch.int32)
    kl = torch.tensor(seqlens, dtype=torch.int32)
    P = 5
    out_s, lse_s = _run(inp, idx, kl, parts=P)
    q, kv, bt, sl = (inp[k].cuda() for k in ("q", "kv_cache", "block_table", "seqlens"))
    meta = mla.decode_metadata(sl, 1, 128, False, P)
    out_d, lse_d = mla.decode(q, kv, bt, sl, inp["softmax_scale"], False, meta, P)
    assert torch.equal(out_s, out_d.cpu()) and torch.equal(lse_s, lse_d.cpu())


def test_sparse_v32_shaped_sampled():
    # DeepSeek-V3.2-shaped: 2048 of 32768 tokens per request, 128 heads
    B, L, k = 8, 32768, 2048
    inp = _case(B, 1, 128, [L] * B, seed=11)
    idx, kl = _lists([L] * B, [k] * B, seed=11)
    out, lse = _run(inp, idx, kl)
    sel = [0, 5, 7]
    sub_out, sub_lse = oracle.decode_sparse(to_np(inp["q"][sel]), inp["kv_cache"].float().numpy(),
                                            inp["block_table"][sel].numpy(), inp["seqlens"][sel].numpy(),
                                            idx[sel].numpy(), kl[sel].numpy(), inp["softmax_scale"])
    compare(out[sel], lse[sel], sub_out, sub_lse, what="sparse V3.2 shape")


def test_sparse_bench_workload_sampled():
    """The sparse workload bench.py times (64 requests, top 2048 of 16384 tokens, the
    workload generator's lists), in the bench's launch configuration; requests 0, 31 and 63
    against the oracle.  Their pages are copied into a compact cache (the block table
    remapped) so that the oracle reads exactly the same rows."""
    import mla_absorbed_decode_gb300 as mla
    w = W.SPARSE
    inp = W.make_inputs(w)
    q, kv, bt, sl = (inp[x].cuda() for x in ("q", "kv_cache", "block_table", "seqlens"))
    idx, kl = inp["indices"], inp["topk_lens"]
    P = mla.num_sm_parts(w.s_q, w.H)
    meta = mla.decode_metadata(kl.cuda(), w.s_q, w.H, w.causal, P)
    out, lse = mla.decode_sparse(q, kv, bt, sl, idx.cuda(), kl.cuda(), w.softmax_scale, w.causal, meta, P)
    assert mla.get_device_status() == 0
    out, lse = out.cpu(), lse.cpu()
    sel = [0, 31, 63]
    npages = (int(sl[0]) + 63) // 64
    rows = inp["block_table"][sel, :npages]
    kv_small = inp["kv_cache"][rows.reshape(-1)].float().numpy()
    bt_small = np.arange(len(sel) * npages, dtype=np.int64).reshape(len(sel), npages)
    ref_out, ref_lse = oracle.decode_sparse(to_np(inp["q"][sel]), kv_small, bt_small, inp["seqlens"][sel].numpy(),
                                            idx[sel].numpy(), kl[sel].numpy(), w.softmax_scale, causal=w.causal)
    compare(out[sel], lse[sel], ref_out, ref_lse, what="sparse bench workload")


def test_sparse_calls_return_promptly():
    """Every call finishes in far less than the kernel's 500 ms bounded-wait limit, for
    batch sizes that give the parts segments of both parities of page counts (a drain
    that waited for an aliased, older phase of a stage barrier once stalled 0.5-1 s at
    exit, with the result still correct)."""
    import mla_absorbed_decode_gb300 as mla
    # ten gathered pages per request at four batch sizes, and the V3.2 shape at half batch
    # (top 2048 of 16384), whose schedule ends parts on segments of one page
    for B, L, k in ((6, 4096, 640), (7, 4096, 640), (9, 4096, 640), (12, 4096, 640), (32, 16384, 2048)):
        inp = _case(B, 1, 128, [L] * B, seed=B)
        idx, kl = _lists([L] * B, [k] * B, seed=B)
        q, kv, bt, sl = (inp[x].cuda() for x in ("q", "kv_cache", "block_table", "seqlens"))
        idx, kl = idx.cuda(), kl.cuda()
        P = mla.num_sm_parts(1, 128)
        meta = mla.decode_metadata(kl, 1, 128, False, P)
        for _ in range(2):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            mla.decode_sparse(q, kv, bt, sl, idx, kl, inp["softmax_scale"], False, meta, P)
            e1.record()
            torch.cuda.synchronize()
            assert mla.get_device_status() == 0
            assert e0.elapsed_time(e1) < 200.0, f"B={B}: {e0.elapsed_time(e1):.1f} ms"


# ------------------------------------------------------------------ FP8 cache --

def _case8(B, s_q, H, seqlens, causal=False, seed=0):
    w = W.Workload("sparse_fp8_case", B=B, s_q=s_q, H=H, causal=causal, fixed_seqlens=tuple(seqlens), kv_fp8=True)
    return make(w, seed=seed)


def _run8(inp, idx, kl, parts=None):
    import mla_absorbed_decode_gb300 as mla
    q, kv, bt, sl = (inp[k].cuda() for k in ("q", "kv_cache", "block_table", "seqlens"))
    B, s_q, H, _ = q.shape
    P = parts or mla.num_sm_parts(s_q, H)
    meta = mla.decode_metadata(kl.cuda(), s_q, H, inp["causal"], P)
    out, lse = mla.decode_sparse_fp8(q, kv, inp["kv_scale"], bt, sl, idx.cuda(), kl.cuda(), inp["softmax_scale"],
                                     inp["causal"], meta, P)
    assert mla.get_device_status() == 0
    return out.cpu(), lse.cpu()


def _ref8(inp, idx, kl):
    return oracle.decode_sparse(to_np(inp["q"]), inp["kv_cache"].numpy(), inp["block_table"].numpy(),
                                inp["seqlens"].numpy(), idx.numpy(), kl.numpy(), inp["softmax_scale"],
                                causal=inp["causal"], kv_scale=inp["kv_scale"])


@pytest.mark.parametrize("H,s_q,causal", [(16, 1, False), (128, 1, False), (128, 2, True), (64, 2, False),
                                           (20, 2, True), (127, 1, False)])
def test_sparse_fp8_small(H, s_q, causal):
    seqlens = [5000, 130, 64, 3000]
    ks = [2048, 130, 1, 777]
    inp = _case8(len(seqlens), s_q, H, seqlens, causal=causal, seed=H + s_q)
    idx, kl = _lists(seqlens, ks, seed=H)
    ref_out, ref_lse = _ref8(inp, idx, kl)
    for parts in (None, 3):
        out, lse = _run8(inp, idx, kl, parts)
        compare(out, lse, ref_out, ref_lse, what=f"sparse fp8 H={H} s_q={s_q} parts={parts}")


def test_sparse_fp8_empty_list_and_unsorted_order():
    seqlens = [300, 900]
    inp = _case8(2, 1, 64, seqlens, seed=5)
    idx, kl = _lists(seqlens, [0, 500], seed=5)
    idx[1, :500] = idx[1, :500][torch.randperm(500, generator=torch.Generator().manual_seed(1))]
    out, lse = _run8(inp, idx, kl)
    ref_out, ref_lse = _ref8(inp, idx, kl)
    compare(out, lse, ref_out, ref_lse, what="sparse fp8 empty/unsorted")
    assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))


def test_sparse_fp8_every_token_listed_matches_the_dense_fp8_kernel():
    # listing every token in order gathers the same rows the dense FP8 kernel loads by TMA;
    # the arithmetic after the load is the same, so the results agree bit for bit
    import mla_absorbed_decode_gb300 as mla
    seqlens = [700, 64, 1]
    inp = _case8(3, 1, 128, seqlens, seed=8)
    idx = torch.full((3, 700), -1, dtype=torch.int32)
    for b, L in enumerate(seqlens):
        idx[b, :L] = torch.arange(L, dtype=torch.int32)
    kl = torch.tensor(seqlens, dtype=torch.int32)
    out_s, lse_s = _run8(inp, idx, kl, parts=2)
    q, kv, bt, sl = (inp[k].cuda() for k in ("q", "kv_cache", "block_table", "seqlens"))
    meta = mla.decode_metadata(sl, 1, 128, False, 2)
    out_d, lse_d = mla.decode_fp8(q, kv, inp["kv_scale"], bt, sl, inp["softmax_scale"], False, meta, 2)
    assert mla.get_device_status() == 0
    assert torch.equal(out_s, out_d.cpu()) and torch.equal(lse_s, lse_d.cpu())


def test_fp8_calls_return_promptly():
    """The same guard for the FP8-cache kernels (four page stages, four q blocks), sparse
    and dense, over batch sizes and part counts that split requests."""
    import mla_absorbed_decode_gb300 as mla
    L, k = 4096, 640
    for B in (6, 7, 9, 12):
        inp = _case8(B, 1, 128, [L] * B, seed=B)
        idx, kl = _lists([L] * B, [k] * B, seed=B)
        q, kv, bt, sl = (inp[x].cuda() for x in ("q", "kv_cache", "block_table", "seqlens"))
        idx, kl = idx.cuda(), kl.cuda()
        P = mla.num_sm_parts(1, 128)
        calls = [("sparse", mla.decode_metadata(kl, 1, 128, False, P), P)]
        for parts in (P, 5):
            calls.append(("dense", mla.decode_metadata(sl, 1, 128, False, parts), parts))
        for kind, meta, parts in calls:
            for _ in range(2):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                if kind == "sparse":
                    mla.decode_sparse_fp8(q, kv, inp["kv_scale"], bt, sl, idx, kl, inp["softmax_scale"], False,
                                          meta, parts)
                else:
                    mla.decode_fp8(q, kv, inp["kv_scale"], bt, sl, inp["softmax_scale"], False, meta, parts)
                e1.record()
                torch.cuda.synchronize()
                assert mla.get_device_status() == 0
                assert e0.elapsed_time(e1) < 200.0, f"{kind} B={B} parts={parts}: {e0.elapsed_time(e1):.1f} ms"
