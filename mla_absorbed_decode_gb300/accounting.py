"""Algorithmic work of absorbed MLA decode: FLOPs and bytes, as the roofline counts them.

Per visible (query, key) pair and head the absorbed path does a 576-deep dot
product for the score and a 512-wide accumulation for the output:
2*(576 + 512) = 2176 FLOPs per head ("MLA 推理：两条计算路径与FlashMLA",
section "谁快", per-pair count of path 2; 278,528 for 128 heads).  Each cached
token is read once per request: 576 bf16 = 1152 bytes (same page, "decode 注意力
变成了计算问题"; "为什么 MLA + MTP 容易吃亏", appendix A: B = b*L*(d_c + d_s)).
Counted bytes add q, out, lse, the used block-table entries and seqlens; page
padding, split partials and metadata are overheads, not algorithmic bytes.

The same page's FLOP counter for both paths (expand vs absorb, per pair and
per token) is restated in ``pair_flops`` / ``fixed_flops`` / ``path_flops``.
"""
from __future__ import annotations

PAGE = 64
D_C = 512      # latent width (kv_lora_rank)
D_R = 64       # shared RoPE key width (qk_rope_head_dim)
D_NOPE = 128   # per-head non-positional q/k width
D_V = 128      # per-head value width
BF16 = 2
FP8 = 1        # an FP8 (E4M3) cache: 576 bytes per token ("MLA 推理：两条计算路径与FlashMLA", exercise 2)


def pair_flops(H: int, absorbed: bool) -> int:
    """FLOPs per (query, key) pair over all heads: QK dot product plus PV accumulation."""
    if absorbed:
        return 2 * H * (D_C + D_R) + 2 * H * D_C
    return 2 * H * (D_NOPE + D_R) + 2 * H * D_V


def fixed_flops(H: int, absorbed: bool) -> int:
    """Per-token fixed cost: expansion of each cached latent (expand) or the two
    per-query projections W_UK / W_UV (absorb)."""
    if absorbed:
        return 2 * H * D_NOPE * D_C + 2 * H * D_C * D_V
    return 2 * D_C * H * (D_NOPE + D_V)


def causal_pairs(n_new: int, n_total: int) -> int:
    """(query, key) pairs when n_new queries follow a cache whose length
    n_total includes them, each seeing only keys up to itself."""
    return n_new * n_total - n_new * (n_new - 1) // 2


def path_flops(n_new: int, n_total: int, H: int = 128):
    """(expand, absorb) FLOPs for n_new new tokens on a cache of n_total tokens."""
    pairs = causal_pairs(n_new, n_total)
    expand = n_total * fixed_flops(H, False) + pairs * pair_flops(H, False)
    absorb = n_new * fixed_flops(H, True) + pairs * pair_flops(H, True)
    return expand, absorb


def crossover_new_tokens(H: int = 128) -> float:
    """New-token count above which expanding wins when the cache is long:
    expansion cost per cached token over the per-pair cost difference."""
    return fixed_flops(H, False) / (pair_flops(H, True) - pair_flops(H, False))


def arithmetic_intensity(H: int = 128, d_c: int = D_C, d_s: int = D_R, b: int = BF16) -> float:
    """FLOP per byte of one-query decode: (2H/b) * (2 d_c + d_s) / (d_c + d_s)."""
    return (2.0 * H / b) * (2 * d_c + d_s) / (d_c + d_s)


def visible(seqlen: int, s_q: int, i: int, causal: bool) -> int:
    if not causal:
        return max(0, seqlen)
    return max(0, min(seqlen, seqlen - s_q + i + 1))


def decode_work(seqlens, s_q: int, H: int, causal: bool, kv_value_bytes: int = BF16):
    """Algorithmic (flops, bytes) of one mla_decode call (kv_value_bytes = FP8: one
    mla_decode_fp8 call; its scale is one number, not counted)."""
    seqlens = [int(x) for x in seqlens]
    B = len(seqlens)
    pairs = sum(visible(L, s_q, i, causal) for L in seqlens for i in range(s_q))
    flops = pairs * H * 2 * ((D_C + D_R) + D_C)
    kv_bytes = sum(max(L, 0) for L in seqlens) * (D_C + D_R) * kv_value_bytes
    rows = B * s_q * H
    q_bytes = rows * (D_C + D_R) * BF16
    out_bytes = rows * D_C * BF16 + rows * 4
    pages = sum((L + PAGE - 1) // PAGE for L in seqlens if L > 0)
    table_bytes = pages * 4 + B * 4
    return flops, kv_bytes + q_bytes + out_bytes + table_bytes


def sparse_decode_work(seqlens, topk_lens, s_q: int, H: int, causal: bool, indices=None, kv_value_bytes: int = BF16):
    """Algorithmic (flops, bytes) of one mla_decode_sparse call: each listed token is
    gathered once per request (1152 bytes) and takes part in every visible pair.
    Without causal masking every query position sees the whole list; with it, position
    i sees the listed positions t <= seqlens[b] - s_q + i (indices needed).  Bytes add
    q, out, lse, the list entries (4 bytes each), one block-table entry per page the
    list touches, and the two per-request lengths.  kv_value_bytes = FP8: 576 bytes per
    listed token (mla_decode_sparse_fp8)."""
    seqlens = [int(x) for x in seqlens]
    topk_lens = [int(x) for x in topk_lens]
    B = len(seqlens)
    pairs = 0
    pages = 0
    for b, (L, k) in enumerate(zip(seqlens, topk_lens)):
        if causal:
            lst = [int(t) for t in indices[b][:k]]
            pairs += sum(sum(1 for t in lst if t < L - s_q + i + 1) for i in range(s_q))
        else:
            pairs += k * s_q
        if indices is not None:
            pages += len({int(t) // PAGE for t in indices[b][:k]})
        else:
            pages += min(k, (L + PAGE - 1) // PAGE)
    flops = pairs * H * 2 * ((D_C + D_R) + D_C)
    kv_bytes = sum(topk_lens) * (D_C + D_R) * kv_value_bytes
    rows = B * s_q * H
    q_bytes = rows * (D_C + D_R) * BF16
    out_bytes = rows * D_C * BF16 + rows * 4
    return flops, kv_bytes + q_bytes + out_bytes + sum(topk_lens) * 4 + pages * 4 + B * 8


def bmm_work(n_tokens: int, H: int, absorb: bool, weight_bytes: int = BF16):
    """(flops, bytes) of q_nope@W_UK (absorb) or o_lat@W_UV (un-absorb) for n_tokens rows;
    weight_bytes = FP8 for E4M3 weights (bmm_fp8; the bf16 activation is read once and
    quantized on chip, so it still counts 2 bytes a value)."""
    flops = 2 * n_tokens * H * D_NOPE * D_C
    w = H * D_NOPE * D_C * weight_bytes
    if absorb:
        io = n_tokens * H * (D_NOPE + D_C) * BF16
    else:
        io = n_tokens * H * (D_C + D_V) * BF16
    return flops, w + io


def extend_work(seqlen: int, T: int, H: int):
    """Algorithmic (flops, bytes) of one chunked extend on the expanded path: every cached
    token's latent is expanded once per head into a 128-value key and a 128-value value
    (2 * 512 * 256 flops), and each visible (new token, cached token) pair costs
    2 * (192 + 128) flops per head ("MLA 推理", the FLOP counter's expanded pair, 82K at
    H = 128); new token i (at position seqlen - T + i) sees seqlen - T + i + 1 tokens.
    Bytes: the cache read once (1152 per token), W_UK and W_UV, q_nope and q_pe in, out and
    lse out; the expanded chunks are intermediates, not algorithmic bytes."""
    pairs = sum(seqlen - T + i + 1 for i in range(T))
    flops = seqlen * H * 2 * D_C * (D_NOPE + D_V) + pairs * H * 2 * (D_NOPE + D_R + D_V)
    nbytes = seqlen * (D_C + D_R) * BF16 + 2 * H * D_NOPE * D_C * BF16 + T * H * (D_NOPE + D_R + D_V) * BF16 + T * H * 4
    return flops, nbytes


def roofline_time(flops: float, nbytes: float, peak_flops: float, peak_bw: float) -> float:
    """max(FLOPs / peak FLOP/s, bytes / peak bytes/s), in seconds."""
    return max(flops / peak_flops, nbytes / peak_bw)
