"""GPU parity of the W_UK / W_UV projections and of the whole chain
(absorb -> decode -> un-absorb) against the expanded, un-absorbed definition."""
import math

import numpy as np
import pytest
import torch

import oracle
from mla_absorbed_decode_gb300 import workloads as W

from _harness import OUT_ABS, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_absorbed_decode_gb300 import build_lib
    build_lib.build()
    yield


def _bf(x):
    return x.to(torch.bfloat16)


def _bmm_bound(ref):
    # one bf16 rounding of an fp32 result: half an ulp is 2^-9 |x|; allow 2^-8 |x| + 1e-3
    return 2.0 ** -8 * np.abs(ref) + 1e-3


@pytest.mark.parametrize("N,H", [(1, 1), (5, 16), (64, 128), (130, 8)])
def test_absorb_q(N, H):
    import mla_absorbed_decode_gb300 as mla
    g = torch.Generator().manual_seed(N * 131 + H)
    q_nope = _bf(torch.randn((N, H, 128), generator=g))
    q_pe = _bf(torch.randn((N, H, 64), generator=g))
    w_uk = _bf(torch.randn((H, 128, 512), generator=g) / math.sqrt(512))
    q = torch.full((N, H, 576), float("nan"), dtype=torch.bfloat16, device="cuda")
    mla.absorb_q(q_nope.cuda(), w_uk.cuda(), q, q_pe=q_pe.cuda())
    assert mla.get_device_status() == 0
    ref = oracle.absorb_q(to_np(q_nope), to_np(w_uk))
    got = to_np(q.cpu())
    assert np.all(np.abs(got[..., :512] - ref) <= _bmm_bound(ref))
    assert torch.equal(q[..., 512:].cpu(), q_pe)


@pytest.mark.parametrize("N,H", [(1, 1), (5, 16), (64, 128), (130, 8)])
def test_absorb_q_with_rope(N, H):
    import mla_absorbed_decode_gb300 as mla
    g = torch.Generator().manual_seed(N * 7 + H)
    q_nope = _bf(torch.randn((N, H, 128), generator=g))
    q_pe = _bf(torch.randn((N, H, 64), generator=g))
    w_uk = _bf(torch.randn((H, 128, 512), generator=g) / math.sqrt(512))
    pos = torch.randint(0, 1 << 17, (N,), generator=g, dtype=torch.int32)
    pos[0] = 0
    if N > 2:
        pos[1], pos[2] = 131071, (1 << 24) - 1    # the largest supported position
    q = torch.full((N, H, 576), float("nan"), dtype=torch.bfloat16, device="cuda")
    mla.absorb_q(q_nope.cuda(), w_uk.cuda(), q, q_pe=q_pe.cuda(), positions=pos.cuda(), rope_theta=10000.0)
    assert mla.get_device_status() == 0
    ref = oracle.assemble_q(to_np(q_nope), to_np(q_pe), to_np(w_uk), positions=pos.numpy(), base=10000.0)
    got = to_np(q.cpu())
    assert np.all(np.abs(got[..., :512] - ref[..., :512]) <= _bmm_bound(ref[..., :512]))
    # the rotation in fp32 on an angle accurate to ~1e-7 rad, then one bf16 rounding
    d = np.abs(got[..., 512:] - ref[..., 512:])
    assert np.all(d <= _bmm_bound(ref[..., 512:])), d.max()
    assert torch.equal(q[0, :, 512:].cpu(), q_pe[0])   # position 0 is the identity, bit for bit


@pytest.mark.parametrize("B,s_q,H,parts", [(1, 1, 16, 1), (64, 1, 128, 76), (37, 2, 128, 76), (700, 1, 16, 148),
                                           (8000, 1, 1, 148)])
@pytest.mark.parametrize("rope", [False, True])
def test_absorb_q_plan_matches_the_separate_calls(B, s_q, H, parts, rope):
    """The absorption with the schedule in its launch gives the two separate calls' q and
    metadata bit for bit (requests of length 0 included; every metadata int is written)."""
    import mla_absorbed_decode_gb300 as mla
    g = torch.Generator().manual_seed(B * 13 + s_q * 7 + H + rope)
    N = B * s_q
    q_nope = _bf(torch.randn((N, H, 128), generator=g)).cuda()
    q_pe = _bf(torch.randn((N, H, 64), generator=g)).cuda()
    w_uk = _bf(torch.randn((H, 128, 512), generator=g) / math.sqrt(512)).cuda()
    seqlens = torch.randint(0, 9000, (B,), generator=g, dtype=torch.int32)
    if B > 1:
        seqlens[0] = 0
    seqlens = seqlens.cuda()
    pos = torch.randint(0, 1 << 20, (N,), generator=g, dtype=torch.int32).cuda() if rope else None
    q1 = torch.full((N, H, 576), float("nan"), dtype=torch.bfloat16, device="cuda")
    mla.absorb_q(q_nope, w_uk, q1, q_pe=q_pe, positions=pos)
    meta1 = mla.decode_metadata(seqlens, s_q, H, False, parts)
    q2 = torch.full((N, H, 576), float("nan"), dtype=torch.bfloat16, device="cuda")
    meta2 = torch.full_like(meta1, -7)
    mla.absorb_q_plan(q_nope, w_uk, q2, seqlens, parts, meta2, q_pe=q_pe, positions=pos)
    assert mla.get_device_status() == 0
    assert torch.equal(q1.view(torch.int16), q2.view(torch.int16))
    assert torch.equal(meta1, meta2)


def test_absorb_q_rope_rejects_bad_arguments():
    import mla_absorbed_decode_gb300 as mla
    N, H = 4, 2
    q_nope = torch.zeros((N, H, 128), dtype=torch.bfloat16, device="cuda")
    q_pe = torch.zeros((N, H, 64), dtype=torch.bfloat16, device="cuda")
    w_uk = torch.zeros((H, 128, 512), dtype=torch.bfloat16, device="cuda")
    q = torch.empty((N, H, 576), dtype=torch.bfloat16, device="cuda")
    pos = torch.zeros(N, dtype=torch.int32, device="cuda")
    for theta in (1.0, 0.5, float("nan"), float("inf")):
        with pytest.raises(mla.MLAError):
            mla.absorb_q(q_nope, w_uk, q, q_pe=q_pe, positions=pos, rope_theta=theta)
    with pytest.raises(mla.MLAError):   # RoPE needs q_pe
        mla.absorb_q(q_nope, w_uk, q, q_pe=None, positions=pos)


@pytest.mark.parametrize("N,H", [(1, 1), (5, 16), (64, 128), (130, 8)])
def test_unabsorb_o(N, H):
    import mla_absorbed_decode_gb300 as mla
    g = torch.Generator().manual_seed(N * 17 + H)
    o_lat = _bf(torch.randn((N, H, 512), generator=g) * 0.1)
    w_uv = _bf(torch.randn((H, 512, 128), generator=g) / math.sqrt(512))
    o = mla.unabsorb_o(o_lat.cuda(), w_uv.cuda())
    assert mla.get_device_status() == 0
    ref = oracle.unabsorb_o(to_np(o_lat), to_np(w_uv))
    got = to_np(o.cpu())
    assert np.all(np.abs(got - ref) <= _bmm_bound(ref))


def _chain(inp, batches=None, positions=None):
    import mla_absorbed_decode_gb300 as mla
    B, s_q, H = inp["q"].shape[:3]
    step = mla.DecodeStep(B, s_q, H, inp["seqlens"].cuda(), inp["causal"], inp["softmax_scale"])
    o = step.run(inp["q_nope"].cuda(), inp["q_pe"].cuda(), inp["w_uk"].cuda(), inp["w_uv"].cuda(),
                 inp["kv_cache"].cuda(), inp["block_table"].cuda(),
                 positions=None if positions is None else positions.cuda())
    assert mla.get_device_status() == 0
    o = o.view(B, s_q, H, 128).cpu()
    sel = list(range(B)) if batches is None else batches
    kv = inp["kv_cache"].float().numpy()
    qn = to_np(inp["q_nope"]).reshape(B, s_q, H, 128)
    qp = to_np(inp["q_pe"])
    if positions is not None:   # the expanded definition sees the rotated q^R
        qp = np.swapaxes(oracle.rope_interleaved(np.swapaxes(qp, 0, 1), positions.numpy()), 0, 1)
    qp = qp.reshape(B, s_q, H, 64)
    ref, ref_lse = oracle.decode_expanded(qn[sel], qp[sel], to_np(inp["w_uk"]), to_np(inp["w_uv"]), kv,
                                          inp["block_table"][sel].numpy(), inp["seqlens"][sel].numpy(),
                                          inp["softmax_scale"], causal=inp["causal"])
    return to_np(o[sel]), ref, step


def test_chain_small_vs_expanded_definition():
    w = W.small_variant(W.V3, B=3, seqlen=700)
    inp = W.make_inputs(w)
    got, ref, _ = _chain(inp)
    d = np.abs(got - ref)
    assert d.max() <= OUT_ABS, d.max()
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= 2e-2


def test_chain_with_rope_vs_expanded_definition():
    w = W.small_variant(W.V3, B=3, seqlen=700)
    inp = W.make_inputs(w)
    positions = inp["seqlens"] - 1   # the new token's position
    got, ref, _ = _chain(inp, positions=positions.to(torch.int32))
    d = np.abs(got - ref)
    assert d.max() <= OUT_ABS, d.max()
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= 2e-2


def test_chain_full_v3_vs_expanded_definition():
    # every request of the full DeepSeek-V3-shaped workload through absorb -> decode ->
    # un-absorb, against the expanded (un-absorbed) definition (~4.4e12 fp64 FLOPs on the host)
    inp = W.make_inputs(W.V3)
    got, ref, _ = _chain(inp)
    d = np.abs(got - ref)
    assert d.max() <= OUT_ABS, d.max()
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= 2e-2
