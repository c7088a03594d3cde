"""mla_decode_noalloc: the decode entry point for callers that cannot allocate.

Some callers cannot hand the library a workspace: an inference engine or plugin
whose memory pool gives out no scratch, or a decode loop that must never call
into the allocator.  mla_decode_noalloc keeps the schedule metadata and the
split partials in a fixed array of device memory inside the library instead.
This test calls it through the C ABI twice in a row, with different requests
(the second call finds the first call's data in the shared array), and checks
each result against mla_decode on the same inputs, within the parity
tolerance, and against the CPU oracle directly.  It sits in a file collected
last so that a failure here does not hide any other test.
"""
import ctypes

import pytest
import torch

from mla_absorbed_decode_gb300 import workloads as W

from _harness import compare, oracle_decode, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_absorbed_decode_gb300 import build_lib
    build_lib.build()
    yield


def _call_noalloc(inp, parts):
    import mla_absorbed_decode_gb300 as mla
    q, kv = inp["q"].cuda(), inp["kv_cache"].cuda()
    bt, sl = inp["block_table"].cuda(), inp["seqlens"].cuda()
    B, s_q, H, _ = q.shape
    out = torch.full((B, s_q, H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, s_q, H), float("nan"), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    st = mla.lib().mla_decode_noalloc(q.data_ptr(), kv.data_ptr(), kv.shape[0], bt.data_ptr(), bt.shape[1],
                                      sl.data_ptr(), B, s_q, H, ctypes.c_float(inp["softmax_scale"]),
                                      int(inp["causal"]), parts, out.data_ptr(), lse.data_ptr(), stream)
    assert st == 0, mla.STATUS_NAMES.get(st, st)
    assert mla.get_device_status() == 0
    return out.cpu(), lse.cpu()


def _call_existing(inp, parts):
    import mla_absorbed_decode_gb300 as mla
    q, kv = inp["q"].cuda(), inp["kv_cache"].cuda()
    bt, sl = inp["block_table"].cuda(), inp["seqlens"].cuda()
    B, s_q, H, _ = q.shape
    meta = mla.decode_metadata(sl, s_q, H, inp["causal"], parts)
    out, lse = mla.decode(q, kv, bt, sl, inp["softmax_scale"], inp["causal"], meta, parts)
    assert mla.get_device_status() == 0
    return out.cpu(), lse.cpu()


def test_noalloc_matches_decode_on_two_calls_in_a_row():
    import mla_absorbed_decode_gb300 as mla
    first = W.make_inputs(W.Workload("na1", B=3, s_q=1, H=128, fixed_seqlens=(900, 64, 3000)), seed=21)
    second = W.make_inputs(W.Workload("na2", B=2, s_q=2, H=64, causal=True, fixed_seqlens=(130, 2000)), seed=22)
    for inp in (first, second):
        B, s_q, H = inp["q"].shape[:3]
        parts = min(mla.num_sm_parts(s_q, H), 12)       # several parts, so requests are split
        out, lse = _call_noalloc(inp, parts)
        ref_out, ref_lse = _call_existing(inp, parts)
        compare(out, lse, to_np(ref_out), to_np(ref_lse), what="noalloc vs mla_decode")
        # and directly against the CPU oracle, within the same parity bounds
        o_out, o_lse, _ = oracle_decode(inp)
        compare(out, lse, o_out, o_lse, what="noalloc vs oracle")


def test_noalloc_refuses_sizes_beyond_its_scratch():
    import mla_absorbed_decode_gb300 as mla
    A = 0x10000   # never dereferenced: the size check comes first
    st = mla.lib().mla_decode_noalloc(A, A, 10, A, 8, A, 4096, 1, 128, ctypes.c_float(0.1), 0, 76, A, A, None)
    assert st == 3   # MLA_ERR_WORKSPACE
