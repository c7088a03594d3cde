"""Launch ordering on the GPU: calls issued back to back on one stream (every library
kernel but the combine may start while the previous kernel still runs, and waits on
griddepcontrol before its first global access), and the whole step recorded in a CUDA
graph and replayed.  Results must equal the same calls issued one at a time."""
import numpy as np
import pytest
import torch

from mla_absorbed_decode_gb300 import workloads as W

from _harness import compare, make, oracle_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_absorbed_decode_gb300 import build_lib
    build_lib.build()
    yield


def test_back_to_back_calls_share_metadata_and_workspace():
    """Three batches with different lengths reuse one metadata and one workspace buffer,
    with no synchronisation between the calls: each schedule must wait for the previous
    decode and combine that read the buffers it overwrites."""
    import mla_absorbed_decode_gb300 as mla
    H = 64
    batches = [[300, 4096, 70], [2000, 1, 129], [64, 65, 5000]]
    inps = [make(W.small_variant(W.TINY, B=3, H=H), seed=i, seqlens=torch.tensor(sl, dtype=torch.int32))
            for i, sl in enumerate(batches)]
    dev = torch.device("cuda")
    parts = mla.num_sm_parts(1, H)
    meta = torch.empty(mla.metadata_size(3, parts) // 4, dtype=torch.int32, device=dev)
    ws = torch.empty(mla.decode_workspace_size(3, 1, H, parts), dtype=torch.uint8, device=dev)
    dev_in = [{k: inp[k].to(dev) for k in ("q", "kv_cache", "block_table", "seqlens")} for inp in inps]
    outs = []
    torch.cuda.synchronize()
    for d, inp in zip(dev_in, inps):
        mla.decode_metadata(d["seqlens"], 1, H, False, parts, out=meta)
        o, l = mla.decode(d["q"], d["kv_cache"], d["block_table"], d["seqlens"], inp["softmax_scale"], False, meta,
                          parts, workspace=ws)
        outs.append((o, l))
    torch.cuda.synchronize()
    assert mla.get_device_status() == 0
    for (o, l), inp in zip(outs, inps):
        ref_out, ref_lse, ref_abs = oracle_decode(inp)
        compare(o, l, ref_out, ref_lse, ref_abs=ref_abs, what=str(inp["seqlens"].tolist()))


def _step_inputs(seed):
    w = W.small_variant(W.V3, B=3, seqlen=700)
    return w, W.make_inputs(w, seed=seed)


def test_graph_replay_equals_eager_and_follows_refilled_inputs():
    import mla_absorbed_decode_gb300 as mla
    dev = torch.device("cuda")
    w, inp = _step_inputs(0)
    _, inp2 = _step_inputs(1)
    kv, bt, sl = (inp[k].to(dev) for k in ("kv_cache", "block_table", "seqlens"))
    qn, qp, wuk, wuv = (inp[k].to(dev) for k in ("q_nope", "q_pe", "w_uk", "w_uv"))
    eager = mla.DecodeStep(w.B, w.s_q, w.H, sl, w.causal, w.softmax_scale, device=dev)
    ref1 = eager.run(qn, qp, wuk, wuv, kv, bt).clone()
    graphed = mla.DecodeStep(w.B, w.s_q, w.H, sl, w.causal, w.softmax_scale, device=dev)
    graphed.capture(qn, qp, wuk, wuv, kv, bt)
    torch.cuda.synchronize()
    graphed.o.zero_()
    got1 = graphed.replay().clone()
    torch.cuda.synchronize()
    assert torch.equal(got1, ref1)
    # refill the captured buffers in place with another batch's q and replay
    qn.copy_(inp2["q_nope"].to(dev))
    qp.copy_(inp2["q_pe"].to(dev))
    ref2 = eager.run(qn, qp, wuk, wuv, kv, bt).clone()
    got2 = graphed.replay().clone()
    torch.cuda.synchronize()
    assert mla.get_device_status() == 0
    assert torch.equal(got2, ref2)
    assert not torch.equal(got1, got2)
    # refill the lengths in place: the captured step recomputes its schedule (inside the
    # absorption's launch) from them, as eager plan() does
    sl.copy_(torch.tensor([700, 1, 333], dtype=torch.int32, device=dev))
    eager.plan()
    ref3 = eager.run(qn, qp, wuk, wuv, kv, bt).clone()
    got3 = graphed.replay().clone()
    torch.cuda.synchronize()
    assert mla.get_device_status() == 0
    assert torch.equal(graphed.metadata, eager.metadata)
    assert torch.equal(got3, ref3)
    assert not torch.equal(got3, got2)
