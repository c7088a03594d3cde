"""GPU parity of the FP8 projections (per-tensor input_to_float8 + bmm_fp8 on kind::f8f6f4
tensor cores) against the oracle's absorb_q_fp8 / unabsorb_o_fp8 through the C ABI.

Both sides quantize the activation with the same float32 steps, so they use the same
codes; what remains is the kernel's fp32 accumulation of exact code products and one bf16
rounding of the result: |delta| <= 2^-8 |ref| + 1e-3 max|ref| elementwise."""
import math

import numpy as np
import pytest
import torch

import oracle
from mla_absorbed_decode_gb300 import workloads as W

from _harness import to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_absorbed_decode_gb300 import build_lib
    build_lib.build()
    yield


W_SCALE = 2.0 ** -9


def _weights_t(g, H, K, J):
    """W[h] is [K, J] ~ N(0, 1/512); returns (bf16 W, its transposed E4M3 codes [H, J, K])."""
    w = (torch.randn((H, K, J), generator=g) / math.sqrt(512)).to(torch.bfloat16)
    codes = (w.float().transpose(1, 2) / W_SCALE).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    return w, codes.contiguous()


def _check(got, ref, what):
    bound = 2.0 ** -8 * np.abs(ref) + 1e-3 * np.abs(ref).max()
    d = np.abs(got - ref)
    assert np.all(d <= bound), f"{what}: max excess {(d - bound).max():.3g}, max|d| {d.max():.3g}"


@pytest.mark.parametrize("N,H,rope", [(1, 1, False), (5, 16, True), (64, 128, True), (200, 4, False)])
def test_absorb_q_fp8(N, H, rope):
    import mla_absorbed_decode_gb300 as mla
    g = torch.Generator().manual_seed(N * 17 + H)
    q_nope = (torch.randn((N, H, 128), generator=g) * 1.7).to(torch.bfloat16)
    q_pe = torch.randn((N, H, 64), generator=g).to(torch.bfloat16)
    _, w_t = _weights_t(g, H, 128, 512)
    pos = torch.randint(0, 1 << 16, (N,), generator=g, dtype=torch.int32) if rope else None
    q = torch.full((N, H, 576), float("nan"), dtype=torch.bfloat16, device="cuda")
    mla.absorb_q_fp8(q_nope.cuda(), w_t.cuda(), W_SCALE, q, q_pe=q_pe.cuda(),
                     positions=None if pos is None else pos.cuda())
    assert mla.get_device_status() == 0
    ref = oracle.assemble_q_fp8(to_np(q_nope), to_np(q_pe), w_t.numpy(), W_SCALE,
                                positions=None if pos is None else pos.numpy())
    got = to_np(q.cpu())
    _check(got[..., :512], ref[..., :512], f"absorb fp8 N={N} H={H}")
    if rope:
        assert np.all(np.abs(got[..., 512:] - ref[..., 512:]) <= 2.0 ** -8 * np.abs(ref[..., 512:]) + 1e-3)
    else:
        assert torch.equal(q[..., 512:].cpu(), q_pe)


@pytest.mark.parametrize("B,s_q,H,parts,rope", [(1, 1, 16, 1, False), (64, 1, 128, 76, True), (37, 2, 128, 76, False),
                                                (8000, 1, 1, 148, True)])
def test_absorb_q_fp8_plan_matches_the_separate_calls(B, s_q, H, parts, rope):
    """The FP8 absorption with the schedule in its amax pass gives the separate calls' q and
    metadata bit for bit (a request of length 0 included)."""
    import mla_absorbed_decode_gb300 as mla
    g = torch.Generator().manual_seed(B * 5 + s_q + H)
    N = B * s_q
    q_nope = (torch.randn((N, H, 128), generator=g) * 1.7).to(torch.bfloat16).cuda()
    q_pe = torch.randn((N, H, 64), generator=g).to(torch.bfloat16).cuda()
    _, w_t = _weights_t(g, H, 128, 512)
    w_t = w_t.cuda()
    seqlens = torch.randint(0, 9000, (B,), generator=g, dtype=torch.int32)
    if B > 1:
        seqlens[0] = 0
    seqlens = seqlens.cuda()
    pos = torch.randint(0, 1 << 16, (N,), generator=g, dtype=torch.int32).cuda() if rope else None
    q1 = torch.full((N, H, 576), float("nan"), dtype=torch.bfloat16, device="cuda")
    mla.absorb_q_fp8(q_nope, w_t, W_SCALE, q1, q_pe=q_pe, positions=pos)
    meta1 = mla.decode_metadata(seqlens, s_q, H, False, parts)
    q2 = torch.full((N, H, 576), float("nan"), dtype=torch.bfloat16, device="cuda")
    meta2 = torch.full_like(meta1, -7)
    mla.absorb_q_fp8_plan(q_nope, w_t, W_SCALE, q2, seqlens, parts, meta2, q_pe=q_pe, positions=pos)
    assert mla.get_device_status() == 0
    assert torch.equal(q1.view(torch.int16), q2.view(torch.int16))
    assert torch.equal(meta1, meta2)


@pytest.mark.parametrize("N,H", [(1, 1), (5, 16), (64, 128), (200, 4)])
def test_unabsorb_o_fp8(N, H):
    import mla_absorbed_decode_gb300 as mla
    g = torch.Generator().manual_seed(N * 29 + H)
    o_lat = (torch.randn((N, H, 512), generator=g) * 0.07).to(torch.bfloat16)   # decode-output scale
    _, w_t = _weights_t(g, H, 512, 128)
    o = torch.full((N, H, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    mla.unabsorb_o_fp8(o_lat.cuda(), w_t.cuda(), W_SCALE, o=o)
    assert mla.get_device_status() == 0
    ref = oracle.unabsorb_o_fp8(to_np(o_lat), w_t.numpy(), W_SCALE)
    _check(to_np(o.cpu()), ref, f"unabsorb fp8 N={N} H={H}")


def test_fp8_projections_of_a_zero_input_and_an_outlier():
    # amax = 0: every code is 0 and the output is exactly 0; one large element sets the scale
    # for the whole tensor (the per-tensor reading), pushing small values into E4M3 subnormals
    import mla_absorbed_decode_gb300 as mla
    g = torch.Generator().manual_seed(3)
    N, H = 6, 8
    _, w_t = _weights_t(g, H, 512, 128)
    o = torch.empty((N, H, 128), dtype=torch.bfloat16, device="cuda")
    mla.unabsorb_o_fp8(torch.zeros((N, H, 512), dtype=torch.bfloat16, device="cuda"), w_t.cuda(), W_SCALE, o=o)
    assert mla.get_device_status() == 0 and torch.all(o == 0)
    x = torch.randn((N, H, 512), generator=g).to(torch.bfloat16)
    x[2, 3, 100] = 3000.0
    mla.unabsorb_o_fp8(x.cuda(), w_t.cuda(), W_SCALE, o=o)
    assert mla.get_device_status() == 0
    _check(to_np(o.cpu()), oracle.unabsorb_o_fp8(to_np(x), w_t.numpy(), W_SCALE), "outlier")


def test_fp8_projections_on_the_bench_workload():
    # the V3 step's projections with the workload generator's FP8 weights, and a reused workspace
    import mla_absorbed_decode_gb300 as mla
    inp = W.make_inputs(W.FP8_PROJ, seqlens=torch.full((W.FP8_PROJ.B,), 64, dtype=torch.int32))
    N, H = inp["q_nope"].shape[:2]
    ws = torch.empty(mla.bmm_fp8_workspace_size(), dtype=torch.uint8, device="cuda")
    pos = torch.full((N,), 4095, dtype=torch.int32)
    q = torch.empty((N, H, 576), dtype=torch.bfloat16, device="cuda")
    mla.absorb_q_fp8(inp["q_nope"].cuda(), inp["w_uk_t_fp8"].cuda(), inp["w_scale"], q, q_pe=inp["q_pe"].cuda(),
                     positions=pos.cuda(), workspace=ws)
    o_lat = (torch.randn((N, H, 512), generator=torch.Generator().manual_seed(5)) * 0.07).to(torch.bfloat16)
    o = mla.unabsorb_o_fp8(o_lat.cuda(), inp["w_uv_t_fp8"].cuda(), inp["w_scale"], workspace=ws)
    assert mla.get_device_status() == 0
    ref_q = oracle.assemble_q_fp8(to_np(inp["q_nope"]), to_np(inp["q_pe"]), inp["w_uk_t_fp8"].numpy(),
                                  inp["w_scale"], positions=pos.numpy())
    _check(to_np(q.cpu())[..., :512], ref_q[..., :512], "V3 absorb fp8")
    _check(to_np(o.cpu()), oracle.unabsorb_o_fp8(to_np(o_lat), inp["w_uv_t_fp8"].numpy(), inp["w_scale"]),
           "V3 unabsorb fp8")
