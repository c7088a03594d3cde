"""Seeded synthetic inputs for absorbed MLA decode.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic, so both the CUDA path and the CPU oracle may use it.

Recipe (the same for every workload; all draws on a CPU torch.Generator seeded
with `seed`, in this fixed order):
  1. seqlens: fixed, or torch.randint(1, max_len + 1, (B,)) for ragged batches;
  2. block table: a random permutation of a pool of ceil(1.03 * total pages)
     pages; request b takes the next ceil(seqlen_b / 64) pool pages in order;
  3. q [B, s_q, H, 576] ~ N(0, 1) in fp32, rounded to bf16 (round-to-nearest-even);
  4. kv [pool, 64, 576] ~ N(0, 1) in fp32;
  5. optional outliers: each slot independently with probability p has its
     whole 576-value row multiplied by a factor (before rounding to bf16);
  6. optional projection inputs: q_nope [B*s_q, H, 128] and q_pe [B*s_q, H, 64]
     ~ N(0, 1); W_UK [H, 128, 512] and W_UV [H, 512, 128] ~ N(0, 1/512) (variance);
  7. optional top-k lists (sparse decode): per request, the first min(topk, L) of a
     random permutation of its positions, sorted ascending (-1 pads the rest).
FP8 cache (kv_fp8): the draws are the same; the cache is stored as E4M3 codes of
kv / kv_scale (clamped to +-448, torch's round-to-nearest conversion) instead of bf16,
with one per-tensor kv_scale.
FP8 projection weights (proj_fp8): the same W_UK / W_UV draws, each head's matrix stored
transposed ([H, 512, 128] and [H, 128, 512], K contiguous) as E4M3 codes of W / w_scale
with one fixed per-tensor w_scale (torch's round-to-nearest conversion, clamped to +-448).
Poison: pool pages no request uses, and slots at or beyond seqlen in a
request's last page, hold NaN (code 0x7F in an FP8 cache); block-table entries past
a request's last page hold -1.  A correct kernel never reads any of them into its result.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

PAGE = 64
D_QK = 576
D_LATENT = 512
D_NOPE = 128
D_ROPE = 64
D_V = 128


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    s_q: int
    H: int
    seqlen: int = 0              # fixed length for every request (0: ragged)
    ragged_max: int = 0          # ragged: seqlens uniform integers in [1, ragged_max]
    causal: bool = False
    outlier_p: float = 0.0
    outlier_scale: float = 1.0
    with_projections: bool = False
    fixed_seqlens: tuple = field(default_factory=tuple)
    topk: int = 0                # sparse decode: each request lists min(topk, L) of its tokens
    kv_fp8: bool = False         # cache stored as FP8 E4M3 codes with one per-tensor scale
    kv_scale: float = 1.0 / 64.0  # dequantized value = code value * kv_scale (N(0,1) draws -> codes within +-448)
    proj_fp8: bool = False       # W_UK / W_UV also given as FP8 E4M3 codes (transposed) with one per-tensor scale
    w_scale: float = 2.0 ** -9   # N(0, 1/512) weights / 2^-9 -> codes of standard deviation ~23, within +-448
    chunk_tokens: int = 0        # chunked extend (expanded path): cached tokens expanded at a time; s_q new tokens

    @property
    def softmax_scale(self) -> float:
        # 1/sqrt(qk_nope + qk_rope) = 1/sqrt(192), the per-head q/k width of the
        # un-absorbed model, which is what the absorbed path must reproduce.
        return 1.0 / math.sqrt(D_NOPE + D_ROPE)

    @property
    def rows(self) -> int:
        return self.s_q * self.H


# The five workloads the parity tests and the bench use.
TINY = Workload("tiny_b2_h16_l256_300", B=2, s_q=1, H=16, fixed_seqlens=(256, 300))
V3 = Workload("deepseek_v3_b64_h128_l4096", B=64, s_q=1, H=128, seqlen=4096, with_projections=True)
RAGGED = Workload("ragged_b128_h128_l1_8192", B=128, s_q=1, H=128, ragged_max=8192)
MTP = Workload("mtp_b64_sq2_causal_h128_l8192", B=64, s_q=2, H=128, seqlen=8192, causal=True)
LONG = Workload("long_b4_h128_l131072_outliers", B=4, s_q=1, H=128, seqlen=131072,
                outlier_p=0.01, outlier_scale=8.0)
# DeepSeek-V3.2-shaped sparse decode (top-k = 2048 of each request's tokens)
SPARSE = Workload("sparse_b64_h128_l16384_top2048", B=64, s_q=1, H=128, seqlen=16384, topk=2048)
# the DeepSeek-V3 shape over an FP8 (E4M3) latent cache
FP8 = Workload("fp8_deepseek_v3_b64_h128_l4096", B=64, s_q=1, H=128, seqlen=4096, with_projections=True,
               kv_fp8=True)
# the DeepSeek-V3.2-shaped sparse decode over an FP8 (E4M3) cache
SPARSE_FP8 = Workload("sparse_fp8_b64_h128_l16384_top2048", B=64, s_q=1, H=128, seqlen=16384, topk=2048, kv_fp8=True)
# the DeepSeek-V3 step with the W_UK / W_UV projections on FP8 weights (bmm_fp8), bf16 cache
FP8_PROJ = Workload("fp8proj_deepseek_v3_b64_h128_l4096", B=64, s_q=1, H=128, seqlen=4096, with_projections=True,
                    proj_fp8=True)
# an extend on the expanded path: 512 new tokens after a 32K-token prefix, chunks of 4096
# ("MLA 推理" exercise 3: a 32K prefix expands to ~2.6 GB per layer at once; chunked, 4096 tokens)
EXTEND = Workload("extend_t512_l32768_h128_chunk4096", B=1, s_q=512, H=128, seqlen=32768, with_projections=True,
                  chunk_tokens=4096)
ALL = (TINY, V3, RAGGED, MTP, LONG, SPARSE, FP8, SPARSE_FP8, FP8_PROJ, EXTEND)
BY_NAME = {w.name: w for w in ALL}


def make_seqlens(w: Workload, g: torch.Generator) -> torch.Tensor:
    if w.fixed_seqlens:
        return torch.tensor(w.fixed_seqlens, dtype=torch.int32)
    if w.ragged_max:
        return torch.randint(1, w.ragged_max + 1, (w.B,), generator=g).to(torch.int32)
    return torch.full((w.B,), w.seqlen, dtype=torch.int32)


def make_inputs(w: Workload, seed: int = 0, seqlens: torch.Tensor | None = None,
                poison: bool = True, max_blocks: int | None = None) -> dict:
    """All CPU tensors of one workload.  Keys:
    q [B,s_q,H,576] bf16, kv_cache [pool,64,576] bf16 (uint8 E4M3 codes with kv_fp8, plus
    kv_scale), block_table [B,max_blocks] int32, seqlens [B] int32, softmax_scale, causal,
    and with projections also
    q_nope [B*s_q,H,128], q_pe [B*s_q,H,64], w_uk [H,128,512], w_uv [H,512,128] (bf16).
    """
    g = torch.Generator().manual_seed(seed)
    sl = make_seqlens(w, g) if seqlens is None else seqlens.to(torch.int32).clone()
    if seqlens is not None and w.ragged_max:
        torch.randint(1, w.ragged_max + 1, (w.B,), generator=g)  # keep the draw order
    B = sl.numel()
    nb = [(int(L) + PAGE - 1) // PAGE if int(L) > 0 else 0 for L in sl]
    used = sum(nb)
    pool = max(1, math.ceil(1.03 * used))
    perm = torch.randperm(pool, generator=g).to(torch.int32)
    mb = max(max(nb) if nb else 0, 1) if max_blocks is None else max_blocks
    bt = torch.full((B, mb), -1, dtype=torch.int32)
    pos = 0
    for b in range(B):
        bt[b, :nb[b]] = perm[pos:pos + nb[b]]
        pos += nb[b]
    q = torch.randn((B, w.s_q, w.H, D_QK), generator=g).to(torch.bfloat16)
    kv = torch.randn((pool, PAGE, D_QK), generator=g)
    if w.outlier_p > 0:
        hit = torch.rand((pool, PAGE), generator=g) < w.outlier_p
        kv[hit] *= w.outlier_scale
    if w.kv_fp8:
        kv = (kv / w.kv_scale).clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
        nan = 0x7F
    else:
        kv = kv.to(torch.bfloat16)
        nan = float("nan")
    if poison:
        in_use = torch.zeros(pool, dtype=torch.bool)
        in_use[perm[:used].long()] = True
        kv[~in_use] = nan
        for b in range(B):
            L = int(sl[b])
            if nb[b] and L % PAGE:
                kv[int(bt[b, nb[b] - 1]), L % PAGE:] = nan
    out = dict(q=q, kv_cache=kv, block_table=bt, seqlens=sl,
               softmax_scale=w.softmax_scale, causal=w.causal)
    if w.kv_fp8:
        out["kv_scale"] = w.kv_scale
    if w.with_projections:
        n = B * w.s_q
        out["q_nope"] = torch.randn((n, w.H, D_NOPE), generator=g).to(torch.bfloat16)
        out["q_pe"] = torch.randn((n, w.H, D_ROPE), generator=g).to(torch.bfloat16)
        std = 1.0 / math.sqrt(512.0)
        out["w_uk"] = (torch.randn((w.H, D_NOPE, D_LATENT), generator=g) * std).to(torch.bfloat16)
        out["w_uv"] = (torch.randn((w.H, D_LATENT, D_V), generator=g) * std).to(torch.bfloat16)
        if w.proj_fp8:
            def codes(t):   # [H, K, J] weights -> [H, J, K] E4M3 codes of t / w_scale
                u = (t.float().transpose(1, 2) / w.w_scale).clamp(-448.0, 448.0)
                return u.to(torch.float8_e4m3fn).view(torch.uint8).contiguous()
            out["w_uk_t_fp8"] = codes(out["w_uk"])
            out["w_uv_t_fp8"] = codes(out["w_uv"])
            out["w_scale"] = w.w_scale
    if w.topk:   # the selector's output: min(topk, L) distinct positions per request, ascending
        idx = torch.full((B, w.topk), -1, dtype=torch.int32)
        kl = torch.zeros(B, dtype=torch.int32)
        for b in range(B):
            L = int(sl[b])
            k = min(w.topk, L)
            idx[b, :k] = torch.randperm(L, generator=g)[:k].sort().values.to(torch.int32)
            kl[b] = k
        out["indices"] = idx
        out["topk_lens"] = kl
    return out


def small_variant(w: Workload, B: int | None = None, seqlen: int | None = None,
                  H: int | None = None) -> Workload:
    """The same workload shape at a size the oracle finishes in seconds."""
    kw = dict(w.__dict__)
    kw["name"] = w.name + "_small"
    if B is not None:
        kw["B"] = B
    if H is not None:
        kw["H"] = H
    if seqlen is not None:
        if w.ragged_max:
            kw["ragged_max"] = seqlen
        elif w.seqlen:
            kw["seqlen"] = seqlen
    if w.fixed_seqlens and B is not None:
        kw["fixed_seqlens"] = tuple(w.fixed_seqlens[i % len(w.fixed_seqlens)] for i in range(B))
    return Workload(**kw)
