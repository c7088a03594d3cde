"""Failure detection on the GPU without a GPU fault.

* A bounded barrier wait that runs out: the test hook withholds the first KV
  page load of every part; every wait on it gives up after its time limit, the
  kernel records MLA_ERR_TIMEOUT and exits cleanly, and the context stays
  usable (the next call is correct).
* A block-table entry outside [0, num_blocks), a top-k list longer than its row
  of indices, or metadata built for a larger batch: the kernel does not read out of
  bounds (the TMA fills the page with zeros), finishes, and records
  MLA_ERR_DEVICE_BOUNDS.
"""
import pytest
import torch

from mla_absorbed_decode_gb300 import workloads as W

from _harness import compare, make, oracle_decode, run_library, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_absorbed_decode_gb300 import build_lib
    build_lib.build()
    yield


def _inputs():
    w = W.Workload("fault", B=2, s_q=1, H=128, fixed_seqlens=(300, 200))
    return make(w, seed=2)


def test_bounded_wait_times_out_and_context_survives():
    import mla_absorbed_decode_gb300 as mla
    inp = _inputs()
    dev = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
    P = 2
    meta = mla.decode_metadata(dev["seqlens"], 1, 128, False, P)
    mla.debug_withhold_first_load(True)
    mla.decode(dev["q"], dev["kv_cache"], dev["block_table"], dev["seqlens"], inp["softmax_scale"], False, meta, P)
    assert mla.get_device_status() == 5          # MLA_ERR_TIMEOUT
    assert mla.get_device_status() == 0          # read-and-clear
    out, lse, _, _ = run_library(inp, parts=P)   # the next call is correct
    ref_out, ref_lse, ref_abs = oracle_decode(inp)
    compare(out, lse, ref_out, ref_lse, what="after timeout")


def test_block_table_out_of_range_is_reported():
    import mla_absorbed_decode_gb300 as mla
    inp = _inputs()
    bt = inp["block_table"].clone()
    bt[1, 1] = inp["kv_cache"].shape[0] + 5      # inside the request's used pages
    dev = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
    dev["block_table"] = bt.cuda()
    P = 2
    meta = mla.decode_metadata(dev["seqlens"], 1, 128, False, P)
    out, lse = mla.decode(dev["q"], dev["kv_cache"], dev["block_table"], dev["seqlens"], inp["softmax_scale"],
                          False, meta, P)
    assert mla.get_device_status() == 6          # MLA_ERR_DEVICE_BOUNDS
    # request 0 does not use the bad entry and is still exact
    ref_out, ref_lse, ref_abs = oracle_decode(inp, [0])
    compare(out[:1].cpu(), lse[:1].cpu(), ref_out, ref_lse, what="request 0 beside a bad entry")


def test_bounded_wait_times_out_fp8_cache():
    # the same withheld load in the FP8-cache kernel (four page stages, four q blocks): the
    # wait runs out, the CTAs drain what they issued, and the next FP8 call is correct
    import mla_absorbed_decode_gb300 as mla
    w = W.Workload("fault_fp8", B=2, s_q=1, H=128, fixed_seqlens=(300, 200), kv_fp8=True)
    inp = make(w, seed=2)
    dev = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
    P = 2
    meta = mla.decode_metadata(dev["seqlens"], 1, 128, False, P)
    mla.debug_withhold_first_load(True)
    mla.decode_fp8(dev["q"], dev["kv_cache"], inp["kv_scale"], dev["block_table"], dev["seqlens"],
                   inp["softmax_scale"], False, meta, P)
    assert mla.get_device_status() == 5          # MLA_ERR_TIMEOUT
    assert mla.get_device_status() == 0
    out, lse, _, _ = run_library(inp, parts=P)
    ref_out, ref_lse, _ = oracle_decode(inp)
    compare(out, lse, ref_out, ref_lse, what="fp8 after timeout")


def test_sparse_list_longer_than_its_index_row_is_reported():
    # topk_lens[b] > index_stride breaks the call's precondition: the kernel reads no
    # entry past the row (the indices here sit inside a larger buffer whose tail holds
    # valid positions, so a stray read would go unreported rather than fault), reports
    # MLA_ERR_DEVICE_BOUNDS, and request 0 keeps its exact result
    import numpy as np
    import oracle
    import mla_absorbed_decode_gb300 as mla
    w = W.Workload("fault_sparse", B=2, s_q=1, H=128, fixed_seqlens=(700, 900))
    inp = make(w, seed=4)
    stride = 128
    rng = np.random.default_rng(4)
    buf = np.zeros(2 * stride + 256, dtype=np.int32)
    buf[:stride] = np.sort(rng.choice(700, size=stride, replace=False))
    buf[stride:2 * stride] = np.sort(rng.choice(900, size=stride, replace=False))
    buf[2 * stride:] = np.arange(256)                    # valid positions of request 1
    kl = torch.tensor([stride, stride + 64], dtype=torch.int32)
    dev = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
    idx_buf = torch.from_numpy(buf).cuda()
    idx = idx_buf[:2 * stride].view(2, stride)
    P = 3
    meta = mla.decode_metadata(kl.cuda(), 1, 128, False, P)
    out, lse = mla.decode_sparse(dev["q"], dev["kv_cache"], dev["block_table"], dev["seqlens"], idx, kl.cuda(),
                                 inp["softmax_scale"], False, meta, P)
    assert mla.get_device_status() == 6          # MLA_ERR_DEVICE_BOUNDS
    ref_out, ref_lse = oracle.decode_sparse(to_np(inp["q"][:1]), inp["kv_cache"].float().numpy(),
                                            inp["block_table"][:1].numpy(), inp["seqlens"][:1].numpy(),
                                            buf[:stride].reshape(1, stride), np.array([stride]), inp["softmax_scale"])
    compare(out[:1].cpu(), lse[:1].cpu(), ref_out, ref_lse, what="sparse request 0 beside an over-long list")


def test_metadata_of_a_larger_batch_is_reported():
    # metadata built for 8 requests handed to a call with 4: the part records that name
    # requests 4..7 are refused on the device (MLA_ERR_DEVICE_BOUNDS) instead of walking
    # past the caller's seqlens, block table and outputs
    import mla_absorbed_decode_gb300 as mla
    w8 = W.Workload("fault_meta8", B=8, s_q=1, H=128, fixed_seqlens=(300, 200, 640, 64, 900, 128, 700, 256))
    inp = make(w8, seed=6)
    P = 6
    meta8 = mla.decode_metadata(inp["seqlens"].cuda(), 1, 128, False, P)
    q4, bt4, sl4 = inp["q"][:4].cuda(), inp["block_table"][:4].cuda(), inp["seqlens"][:4].cuda()
    mla.decode(q4, inp["kv_cache"].cuda(), bt4, sl4, inp["softmax_scale"], False, meta8, P)
    assert mla.get_device_status() == 6          # MLA_ERR_DEVICE_BOUNDS
    assert mla.get_device_status() == 0
