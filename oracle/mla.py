"""Plain float64 restatement of weight-absorbed MLA decode (test infrastructure only).

Sources (web pages, cited by title and section):

[MLA-paths]  "MLA 推理：两条计算路径与 FlashMLA" (ai-infra-handbooks, serving/moe/mla),
             section "两条等价的路径" (the score equation s = q^N·W_UK^T c + q^R·k^R,
             path 1 = expand, path 2 = absorb), its worked tiny example, and section
             "decode 注意力变成了计算问题" (split-KV partial results merged at the end).
[DSV2-MLA]   "DeepSeekV2之MLA", section 4.3 (decode attention is an MQA with one
             KV head, key width kv_lora_rank + rope = 576, value width 512) and
             section 4.5 (q_nope @ w_kc into the latent, attention, then @ w_vc).
[AI-note]    "为什么 MLA + MTP 容易吃亏？从 Arithmetic Intensity 看 Attention",
             sections 3.1 (K-side absorption), 3.2 (V-side absorption),
             section 8 (S query positions share one KV read) and appendix A
             (the 64-dim RoPE key takes part in the score only, it has no value).

Readings taken where the pages are silent:
* lse is the natural log of the sum of exp of the *scaled* scores.
* With s_q > 1 and causal masking, seqlens counts the s_q new tokens and new
  token i (0 = earliest) sees tokens t <= seqlen - s_q + i  ([MLA-paths],
  FLOP counter: its key count takes in the new tokens, pairs = q*k - q(q-1)/2).
* A query row with no visible token has out = 0 and lse = -inf.
* Token t of request b lives at kv_cache[block_table[b, t // 64], t % 64]; the
  page size 64 is the one FlashMLA uses ([MLA-paths], FlashMLA paragraph).
"""
from __future__ import annotations

import math

import numpy as np

PAGE = 64          # tokens per KV page
D_LATENT = 512     # latent c (also the value)
D_ROPE = 64        # shared RoPE key k^R
D_QK = D_LATENT + D_ROPE  # 576: width of the absorbed key / query


def e4m3_value(code: int) -> float:
    """The number an FP8 E4M3 byte stands for (the "e4m3fn" encoding of FP8 KV caches).

    Bit 7 is the sign, bits 6..3 the exponent e (bias 7), bits 2..0 the mantissa m:
        e > 0:  (-1)^s * (1 + m/8) * 2^(e - 7)
        e = 0:  (-1)^s * (m/8) * 2^-6            (subnormal)
    The two codes with e = 15 and m = 7 are NaN; there is no infinity, so the largest
    finite magnitude is 1.75 * 2^8 = 448.
    """
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** -6
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


E4M3_VALUES = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)


def dequantize_e4m3(codes, scale: float) -> np.ndarray:
    """Cached FP8 values as float64: the code's E4M3 value times the per-tensor scale.

    [MLA-paths], exercise 2 ("FP8 的 KV Cache"): a token's 576 latent values are stored
    one byte each, with scale factors beside them.  The reading taken here is one scale
    for the whole cache, the per-tensor convention of the FP8 bmm in the SGLang page
    (bmm_fp8 with a scale per operand).
    """
    return E4M3_VALUES[np.asarray(codes, dtype=np.uint8)] * float(scale)


def gather_request(kv_cache: np.ndarray, block_row: np.ndarray, n_tokens: int, kv_scale=None) -> np.ndarray:
    """Rows 0..n_tokens-1 of one request's latent cache, as float64 [n_tokens, 576].

    kv_cache is [num_blocks, 64, 576]; block_row is that request's row of the
    block table.  Token t sits in page block_row[t // 64] at slot t % 64.  With
    kv_scale given, the cache holds E4M3 codes (uint8) and each gathered row is
    dequantized (dequantize_e4m3).
    """
    t = np.arange(n_tokens)
    pages = np.asarray(block_row)[t // PAGE]
    rows = np.asarray(kv_cache[pages, t % PAGE])
    if kv_scale is not None:
        return dequantize_e4m3(rows, kv_scale)
    return np.asarray(rows, dtype=np.float64)


def visible_tokens(seqlen: int, s_q: int, i: int, causal: bool) -> int:
    """How many cached tokens query position i (0 = earliest new token) attends to."""
    if not causal:
        return int(seqlen)
    return max(0, min(int(seqlen), int(seqlen) - s_q + i + 1))


def decode_absorbed(q, kv_cache, block_table, seqlens, softmax_scale, causal=False, with_abs=False,
                    kv_scale=None):
    """The absorbed decode definition: an MQA with a 576-wide key and 512-wide value.

    For every request b, query position i and head h, with n = visible tokens:
        s_t   = softmax_scale * <q[b,i,h,:576], kv_t[:576]>         t < n
        lse   = ln sum_t exp(s_t)
        out   = sum_t exp(s_t - lse) * kv_t[:512]
    ([MLA-paths] path 2; [DSV2-MLA] 4.3; [AI-note] 3.1-3.2 and appendix A.)

    q: [B, s_q, H, 576]; kv_cache: [num_blocks, 64, 576]; block_table: [B, max_blocks];
    seqlens: [B].  Returns out [B, s_q, H, 512] and lse [B, s_q, H], float64.
    The softmax is evaluated with its maximum subtracted, which changes only rounding.
    With with_abs=True it also returns out_abs = sum_t p_t |kv_t[:512]|, the
    attention-weighted magnitude of the values, which sizes the rounding error of
    a kernel that rounds p_t to bf16 (test tolerance, not part of the method).
    With kv_scale given, kv_cache holds FP8 E4M3 codes and kv_t is the dequantized
    row (gather_request); see decode_fp8.
    """
    q = np.asarray(q, dtype=np.float64)
    B, s_q, H, dq = q.shape
    assert dq == D_QK
    out = np.zeros((B, s_q, H, D_LATENT))
    out_abs = np.zeros((B, s_q, H, D_LATENT)) if with_abs else None
    lse = np.full((B, s_q, H), -np.inf)
    for b in range(B):
        L = int(seqlens[b])
        if L <= 0:
            continue
        kv = gather_request(kv_cache, block_table[b], L, kv_scale)
        for i in range(s_q):
            n = visible_tokens(L, s_q, i, causal)
            if n == 0:
                continue
            s = softmax_scale * (q[b, i] @ kv[:n].T)          # [H, n]
            m = s.max(axis=1, keepdims=True)
            e = np.exp(s - m)
            z = e.sum(axis=1, keepdims=True)
            lse[b, i] = (m + np.log(z))[:, 0]
            out[b, i] = (e / z) @ kv[:n, :D_LATENT]
            if with_abs:
                out_abs[b, i] = (e / z) @ np.abs(kv[:n, :D_LATENT])
    if with_abs:
        return out, lse, out_abs
    return out, lse


def decode_fp8(q, kv_codes, kv_scale, block_table, seqlens, softmax_scale, causal=False, with_abs=False):
    """Absorbed decode over an FP8 (E4M3) latent cache with one per-tensor scale.

    [MLA-paths], FlashMLA paragraph (the kernel supports an FP8 KV cache) and exercise 2
    (576 bytes per cached token plus scale factors): the attention is the one of
    decode_absorbed, over kv_t = dequantize_e4m3(kv_codes[page, slot], kv_scale);
    q stays bf16.  kv_codes: [num_blocks, 64, 576] uint8.
    """
    return decode_absorbed(q, kv_codes, block_table, seqlens, softmax_scale, causal, with_abs, kv_scale=kv_scale)


def decode_sparse(q, kv_cache, block_table, seqlens, indices, topk_lens, softmax_scale, causal=False,
                  with_abs=False, kv_scale=None):
    """Sparse (top-k) absorbed decode: the same attention, over a selected list of tokens.

    [AI-note] section 6 ("Sparse attention 把方向反过来"): a selector picks k of the L
    cached latents (DeepSeek-V3.2's DSA, index_topk = 2048); they are gathered by
    index and the scores and the weighted sum run over those k only.  For request b
    the list is indices[b, 0:topk_lens[b]] (token positions, each in [0, seqlens[b]),
    looked up through the block table as in the dense case); with causal masking query
    position i keeps only listed tokens t <= seqlens[b] - s_q + i:
        s_t = softmax_scale * <q[b,i,h,:576], kv_t[:576]>,  t listed and visible
        lse = ln sum_t exp(s_t),   out = sum_t exp(s_t - lse) * kv_t[:512]
    A listed token counts once per listing.  Returns out [B, s_q, H, 512], lse [B, s_q, H].
    With kv_scale given, kv_cache holds FP8 E4M3 codes and kv_t is the dequantized row
    (dequantize_e4m3), as in decode_fp8.
    """
    q = np.asarray(q, dtype=np.float64)
    B, s_q, H, dq = q.shape
    assert dq == D_QK
    out = np.zeros((B, s_q, H, D_LATENT))
    out_abs = np.zeros((B, s_q, H, D_LATENT)) if with_abs else None
    lse = np.full((B, s_q, H), -np.inf)
    for b in range(B):
        sel = np.asarray(indices[b][: int(topk_lens[b])], dtype=np.int64)
        L = int(seqlens[b])
        if sel.size == 0:
            continue
        assert sel.min() >= 0 and sel.max() < L
        rows = np.asarray(kv_cache[np.asarray(block_table[b])[sel // PAGE], sel % PAGE])
        kv = dequantize_e4m3(rows, kv_scale) if kv_scale is not None else np.asarray(rows, dtype=np.float64)
        for i in range(s_q):
            keep = sel < visible_tokens(L, s_q, i, causal)
            if not keep.any():
                continue
            s = softmax_scale * (q[b, i] @ kv[keep].T)          # [H, kept]
            m = s.max(axis=1, keepdims=True)
            e = np.exp(s - m)
            z = e.sum(axis=1, keepdims=True)
            lse[b, i] = (m + np.log(z))[:, 0]
            out[b, i] = (e / z) @ kv[keep, :D_LATENT]
            if with_abs:
                out_abs[b, i] = (e / z) @ np.abs(kv[keep, :D_LATENT])
    if with_abs:
        return out, lse, out_abs
    return out, lse


def absorb_q(q_nope, w_uk):
    """q_lat[b, h, :] = q_nope[b, h, :] @ W_UK[h]   ([DSV2-MLA] 4.5, "q_nope @ w_kc").

    q_nope: [N, H, 128]; w_uk: [H, 128, 512] -> [N, H, 512] float64.
    """
    q_nope = np.asarray(q_nope, dtype=np.float64)
    w_uk = np.asarray(w_uk, dtype=np.float64)
    return np.einsum("nhd,hdc->nhc", q_nope, w_uk)


def assemble_q(q_nope, q_pe, w_uk, positions=None, base=10000.0):
    """The decode query of the absorbed path: q[n, h, 0:512] = q_nope[n, h] @ W_UK[h] and
    q[n, h, 512:576] = q_pe[n, h], rotated by RoPE at positions[n] when positions is given.

    ([DSV2-MLA] 4.5: the absorbed q_nope goes into the first kv_lora_rank values, the
    RoPE'd q_pe into the last 64; the rotation is the decoupled RoPE of the [MLA-paths]
    tiny example, rope_interleaved below.)  q_nope [N, H, 128], q_pe [N, H, 64],
    w_uk [H, 128, 512], positions [N] -> [N, H, 576] float64.
    """
    q_lat = absorb_q(q_nope, w_uk)
    pe = np.asarray(q_pe, dtype=np.float64)
    if positions is not None:
        pe = np.swapaxes(rope_interleaved(np.swapaxes(pe, 0, 1), positions, base), 0, 1)   # rows = tokens
    return np.concatenate([q_lat, pe], axis=-1)


def unabsorb_o(o_lat, w_uv):
    """o[b, h, :] = o_lat[b, h, :] @ W_UV[h]   ([DSV2-MLA] 4.5, "attn_output @ w_vc").

    o_lat: [N, H, 512]; w_uv: [H, 512, 128] -> [N, H, 128] float64.
    """
    o_lat = np.asarray(o_lat, dtype=np.float64)
    w_uv = np.asarray(w_uv, dtype=np.float64)
    return np.einsum("nhc,hcd->nhd", o_lat, w_uv)


def decode_expanded(q_nope, q_pe, w_uk, w_uv, kv_cache, block_table, seqlens, softmax_scale,
                    causal=False, batches=None, head_chunk=16):
    """The expanded (un-absorbed) definition: per-head K and V built from the latent.

    For head h and cached token t with latent c_t = kv_t[:512] and RoPE key
    k^R_t = kv_t[512:576]:
        k_{h,t} = [ W_UK[h] c_t  (128) , k^R_t (64) ]
        v_{h,t} =   W_UV[h]^T c_t (128)
        s       = softmax_scale * <[q_nope, q_pe], k_{h,t}>,   o = softmax(s) . v
    ([MLA-paths] path 1; [AI-note] 3.1-3.2; the orientation of W_UK / W_UV is the
    bmm one of [DSV2-MLA] 4.5: q_lat = q_nope @ W_UK[h], o = o_lat @ W_UV[h].)

    q_nope: [B, s_q, H, 128], q_pe: [B, s_q, H, 64], w_uk: [H, 128, 512],
    w_uv: [H, 512, 128].  Returns o [B, s_q, H, 128] (rows of requests not in
    `batches` stay zero) and lse [B, s_q, H].
    """
    q_nope = np.asarray(q_nope, dtype=np.float64)
    q_pe = np.asarray(q_pe, dtype=np.float64)
    w_uk = np.asarray(w_uk, dtype=np.float64)
    w_uv = np.asarray(w_uv, dtype=np.float64)
    B, s_q, H, _ = q_nope.shape
    dv = w_uv.shape[2]
    o = np.zeros((B, s_q, H, dv))
    lse = np.full((B, s_q, H), -np.inf)
    for b in (range(B) if batches is None else batches):
        L = int(seqlens[b])
        if L <= 0:
            continue
        kv = gather_request(kv_cache, block_table[b], L)
        c, k_r = kv[:, :D_LATENT], kv[:, D_LATENT:]
        for h0 in range(0, H, head_chunk):
            hs = slice(h0, min(H, h0 + head_chunk))
            k_n = np.matmul(c[None], np.transpose(w_uk[hs], (0, 2, 1)))   # [h, L, 128]
            v = np.matmul(c[None], w_uv[hs])                              # [h, L, 128]
            for i in range(s_q):
                n = visible_tokens(L, s_q, i, causal)
                if n == 0:
                    continue
                s = np.einsum("hd,hld->hl", q_nope[b, i, hs], k_n[:, :n]) + q_pe[b, i, hs] @ k_r[:n].T
                s *= softmax_scale
                m = s.max(axis=1, keepdims=True)
                e = np.exp(s - m)
                z = e.sum(axis=1, keepdims=True)
                lse[b, i, hs] = (m + np.log(z))[:, 0]
                o[b, i, hs] = np.einsum("hl,hld->hd", e / z, v[:, :n])
    return o, lse


def lse_merge(o_parts, lse_parts):
    """Merge attention results over disjoint key sets by log-sum-exp.

    ([MLA-paths]: split-KV / flash-decoding computes each KV segment on its own
    SM and merges the partial results; the chunked-prefix path merges chunks
    "by LSE", the same way as context parallelism.)
        lse = ln sum_k exp(lse_k),   o = sum_k exp(lse_k - lse) * o_k
    o_parts: [K, ..., D]; lse_parts: [K, ...].  Parts with lse = -inf carry no
    weight; if every part is empty the result is o = 0, lse = -inf.
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    m = lse_parts.max(axis=0)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    w = np.where(np.isfinite(lse_parts), np.exp(lse_parts - m_safe), 0.0)
    z = w.sum(axis=0)
    lse = np.where(finite, m_safe + np.log(np.where(finite, z, 1.0)), -np.inf)
    coef = np.where(finite, w / np.where(finite, z, 1.0), 0.0)
    o = np.einsum("k...,k...d->...d", coef, o_parts)
    return o, lse


def decode_bruteforce(q_row, keys, softmax_scale):
    """Single query row against a handful of keys, in pure Python loops.

    q_row: 576 numbers; keys: list of 576-number rows.  Returns (out[512], lse).
    No maximum is subtracted: exp is applied to the raw scaled scores, so this
    is only for small, moderate inputs (it is the textbook formula, as is).
    """
    scores = []
    for k in keys:
        acc = 0.0
        for a, bb in zip(q_row, k):
            acc += float(a) * float(bb)
        scores.append(softmax_scale * acc)
    weights = [math.exp(s) for s in scores]
    z = sum(weights)
    out = [0.0] * D_LATENT
    for w, k in zip(weights, keys):
        for d in range(D_LATENT):
            out[d] += (w / z) * float(k[d])
    return out, math.log(z)


def rope_interleaved(x, positions, base=10000.0):
    """Rotate adjacent pairs (x[2j], x[2j+1]) by angle pos * base^(-2j/R).

    ([MLA-paths] tiny example, its rope helper: angle = pos / 10000^(2j/R), the
    rotated pairs are written back interleaved.)  x: [..., T, R]; positions: [T].
    """
    x = np.asarray(x, dtype=np.float64)
    R = x.shape[-1]
    j = np.arange(R // 2, dtype=np.float64)
    ang = np.asarray(positions, dtype=np.float64)[:, None] * base ** (-2.0 * j / R)   # [T, R/2]
    cos, sin = np.cos(ang), np.sin(ang)
    x0, x1 = x[..., 0::2], x[..., 1::2]
    y = np.empty_like(x)
    y[..., 0::2] = x0 * cos - x1 * sin
    y[..., 1::2] = x0 * sin + x1 * cos
    return y


def tiny_full_mla(seed=0, T=6, D=64, H=4, NOPE=8, ROPE=4, DV=8, DC=16):
    """A tiny full MLA layer with decoupled RoPE, evaluated both ways.

    [MLA-paths] section "两条等价的路径" states the score of head h between query
    token i and cached token j as
        s = q^N_{h,i} . k^N_{h,j} + q^R_{h,i} . k^R_j,   k^N_{h,j} = U_k[h] c_j,
    with c_j the cached latent (DC values) and k^R_j the shared RoPE key (ROPE values),
    and the value as v_{h,j} = U_v[h] c_j.  Since q^N . (U_k c) = (U_k^T q^N) . c, the
    same numbers come out of
      * path 1 (expand): build k^N_{h,j} and v_{h,j} for every cached token, then
        ordinary attention;
      * path 2 (absorb): move q^N into the latent space once per query token, score
        against c_j directly, sum p_j c_j in the latent space and apply U_v[h] last.
    Each head's outputs (DV values) are concatenated and projected back to D.  The
    page checks the two paths with allclose and counts the cached numbers per token
    (per-head K and V against c plus k^R); those are the claims kept here.  Weights
    are seeded Gaussians scaled by 1/sqrt(fan-in); prefill-style causal masking (token
    i sees j <= i); softmax scale 1/sqrt(NOPE + ROPE); RoPE at positions 0..T-1.
    Returns y_expand, y_absorb ([T, D]) and the per-token cache counts.
    """
    rng = np.random.default_rng(seed)

    def gauss(rows, cols):   # a (rows x cols) map applied as M @ x, scaled by its fan-in
        return rng.standard_normal((rows, cols)) / math.sqrt(cols)

    x = rng.standard_normal((T, D))                      # hidden states of the T tokens
    to_latent, to_rope_key = gauss(DC, D), gauss(ROPE, D)
    heads = [dict(q_n=gauss(NOPE, D), q_r=gauss(ROPE, D), u_k=gauss(NOPE, DC), u_v=gauss(DV, DC))
             for _ in range(H)]
    out_proj = gauss(D, H * DV)
    pos = np.arange(T)
    scale = 1.0 / math.sqrt(NOPE + ROPE)

    latent = np.stack([to_latent @ x[t] for t in range(T)])                        # cached: c_j
    rope_key = rope_interleaved(np.stack([to_rope_key @ x[t] for t in range(T)]), pos)   # cached: k^R_j

    def probabilities(scores):   # softmax over the visible tokens, maximum subtracted
        e = np.exp(np.asarray(scores) - max(scores))
        return e / e.sum()

    concat = {"expand": np.zeros((T, H * DV)), "absorb": np.zeros((T, H * DV))}
    for h, w in enumerate(heads):
        qn_all = np.stack([w["q_n"] @ x[t] for t in range(T)])
        qr_all = rope_interleaved(np.stack([w["q_r"] @ x[t] for t in range(T)]), pos)
        cols = slice(h * DV, (h + 1) * DV)
        for i in range(T):
            qn, qr = qn_all[i], qr_all[i]
            # path 1: per-head keys and values expanded from the latent
            s1 = [scale * (qn @ (w["u_k"] @ latent[j]) + qr @ rope_key[j]) for j in range(i + 1)]
            p1 = probabilities(s1)
            concat["expand"][i, cols] = sum(p1[j] * (w["u_v"] @ latent[j]) for j in range(i + 1))
            # path 2: the query moves into the latent space; the output leaves it at the end
            q_lat = w["u_k"].T @ qn
            s2 = [scale * (q_lat @ latent[j] + qr @ rope_key[j]) for j in range(i + 1)]
            p2 = probabilities(s2)
            concat["absorb"][i, cols] = w["u_v"] @ sum(p2[j] * latent[j] for j in range(i + 1))
    return {
        "y_expand": concat["expand"] @ out_proj.T,
        "y_absorb": concat["absorb"] @ out_proj.T,
        "cache_per_token_mha": H * (NOPE + ROPE) + H * DV,
        "cache_per_token_mla": DC + ROPE,
    }


# ------------------------------------------------------- FP8 projections (bmm_fp8) --
# [SGL-compile] "SGLang v0.3 MLA / torch.compile", the weight-absorption code walk-through:
# with FP8 weights the absorption runs as
#     x_val, x_scale = input_to_float8(x)            (x = q_nope, or the attention output)
#     y = bmm_fp8(x_val, w, x_scale, w_scale) -> bf16
# one scale per operand.  The page shows the calls, not their bodies; the reading taken
# here is the plain per-tensor one: the activation's scale maps its largest magnitude onto
# E4M3's largest finite value, 448, and the product is the float64 sum of the decoded
# codes times both scales.  The quantization is done in float32 (the scale's reciprocal
# multiplies each float32 value, then one rounding to E4M3), so that a kernel doing the same
# float32 steps reaches the same codes.

E4M3_MAX = 448.0
_E4M3_POS = E4M3_VALUES[:127]          # codes 0x00..0x7E: 0, the subnormals, the normals up to 448


def e4m3_round(v) -> np.ndarray:
    """E4M3 codes (uint8) of float values: the nearest representable value, ties to the
    even code (mantissa bit 0 clear), magnitudes of 448 and above saturated to 448, the sign
    kept (negative values that round to zero give -0, 0x80), NaN to the NaN code 0x7F."""
    v = np.asarray(v, dtype=np.float64)
    mag = np.minimum(np.abs(v), E4M3_MAX)
    hi = np.clip(np.searchsorted(_E4M3_POS, mag, side="left"), 0, 126)   # first code with value >= mag
    lo = np.clip(hi - 1, 0, 126)
    d_hi = _E4M3_POS[hi] - mag
    d_lo = mag - _E4M3_POS[lo]
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (lo % 2 == 0))
    code = np.where(pick_lo, lo, hi).astype(np.uint8)
    code = np.where(np.signbit(v), code | 0x80, code)   # the sign bit is kept, also on values rounding to zero
    return np.where(np.isnan(v), np.uint8(0x7F), code).astype(np.uint8)


def input_to_float8(x):
    """Per-tensor dynamic FP8 quantization of an activation tensor (the page's
    input_to_float8): amax = max |x| over the whole tensor; in float32,
    inv = 448 / amax and scale = amax / 448 (both 1 when amax = 0); codes =
    e4m3_round(float32(x) * inv).  Returns (codes uint8, scale float); x ~= codes' values * scale."""
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.float32(np.max(np.abs(x32))) if x32.size else np.float32(0.0)
    if amax > 0:
        inv = np.float32(E4M3_MAX) / amax
        scale = amax / np.float32(E4M3_MAX)
    else:
        inv = np.float32(1.0)
        scale = np.float32(1.0)
    return e4m3_round((x32 * inv).astype(np.float32)), float(scale)


def bmm_fp8(x_codes, x_scale, w_t_codes, w_scale):
    """Per-head product of FP8 operands (the page's bmm_fp8 with one scale per operand):
        y[n, h, j] = sum_k e4m3(x[n, h, k]) * e4m3(w_t[h, j, k]) * x_scale * w_scale
    x_codes [N, H, K] uint8, w_t_codes [H, J, K] uint8 (each head's weight stored with its K
    values contiguous: W[h] transposed).  Returns float64 [N, H, J]."""
    xv = E4M3_VALUES[np.asarray(x_codes, dtype=np.uint8)]
    wv = E4M3_VALUES[np.asarray(w_t_codes, dtype=np.uint8)]
    return np.einsum("nhk,hjk->nhj", xv, wv) * (float(x_scale) * float(w_scale))


def absorb_q_fp8(q_nope, w_uk_t_codes, w_uk_scale):
    """q_lat = bmm_fp8(input_to_float8(q_nope), W_UK) ([SGL-compile]; [DSV2-MLA] 4.5):
    q_nope [N, H, 128] -> [N, H, 512] float64; w_uk_t_codes [H, 512, 128] (W_UK[h]^T)."""
    codes, scale = input_to_float8(q_nope)
    return bmm_fp8(codes, scale, w_uk_t_codes, w_uk_scale)


def assemble_q_fp8(q_nope, q_pe, w_uk_t_codes, w_uk_scale, positions=None, base=10000.0):
    """The decode query with the FP8 absorption: [absorb_q_fp8(q_nope), q_pe rotated by RoPE
    at positions (copied when positions is None)] -> [N, H, 576] float64 (as assemble_q)."""
    q_lat = absorb_q_fp8(q_nope, w_uk_t_codes, w_uk_scale)
    pe = np.asarray(q_pe, dtype=np.float64)
    if positions is not None:
        pe = np.swapaxes(rope_interleaved(np.swapaxes(pe, 0, 1), positions, base), 0, 1)
    return np.concatenate([q_lat, pe], axis=-1)


def unabsorb_o_fp8(o_lat, w_uv_t_codes, w_uv_scale):
    """o = bmm_fp8(input_to_float8(o_lat), W_UV) ([SGL-compile]; [DSV2-MLA] 4.5):
    o_lat [N, H, 512] -> [N, H, 128] float64; w_uv_t_codes [H, 128, 512] (W_UV[h]^T)."""
    codes, scale = input_to_float8(o_lat)
    return bmm_fp8(codes, scale, w_uv_t_codes, w_uv_scale)


# --------------------------------------------- chunked expanded extend (MHA_CHUNKED_KV) --
# [MLA-paths] end of section "两条等价的路径" and exercise 3: with a long cached prefix, an
# extend (T new tokens after P cached ones) runs on the expanded path with the prefix
# expanded chunk by chunk -- per head K = [W_UK c, k^R] and V = W_UV^T c for the chunk's
# tokens only -- attention of the new tokens to each chunk on its own, and the per-chunk
# results merged by LSE (the merge of context parallelism), so that the whole expanded
# prefix (~80 KB a token) never exists at once.

def expand_chunk(kv_rows, w_uk, w_uv):
    """The expanded keys and values of a run of cached rows ([MLA-paths] path 1):
    k_nope[h, t] = W_UK[h] c_t (128), k_pe[t] = k^R_t (64, shared by the heads),
    v[h, t] = W_UV[h]^T c_t (128).  kv_rows [n, 576]; returns k_nope [H, n, 128],
    k_pe [n, 64], v [H, n, 128] float64."""
    c = np.asarray(kv_rows, dtype=np.float64)[:, :D_LATENT]
    k_pe = np.asarray(kv_rows, dtype=np.float64)[:, D_LATENT:]
    k_nope = np.einsum("hdc,tc->htd", np.asarray(w_uk, dtype=np.float64), c)
    v = np.einsum("tc,hcd->htd", c, np.asarray(w_uv, dtype=np.float64))
    return k_nope, k_pe, v


def attend_chunk(q_nope, q_pe, k_nope, k_pe, v, key_pos, query_pos, softmax_scale):
    """Multi-head attention of T queries to one expanded chunk, causal by position: query i
    (at position query_pos[i]) sees key t if key_pos[t] <= query_pos[i].  q_nope [T, H, 128],
    q_pe [T, H, 64]; k_nope [H, n, 128], k_pe [n, 64], v [H, n, 128].  Returns the chunk's
    normalised output o [T, H, 128] and lse [T, H] (o = 0, lse = -inf for a query that sees
    no key of the chunk)."""
    q_nope = np.asarray(q_nope, dtype=np.float64)
    q_pe = np.asarray(q_pe, dtype=np.float64)
    T, H, _ = q_nope.shape
    o = np.zeros((T, H, v.shape[2]))
    lse = np.full((T, H), -np.inf)
    for i in range(T):
        seen = np.asarray(key_pos) <= query_pos[i]
        if not seen.any():
            continue
        s = softmax_scale * (np.einsum("hd,htd->ht", q_nope[i], k_nope[:, seen]) + q_pe[i] @ k_pe[seen].T)
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        z = e.sum(axis=1, keepdims=True)
        lse[i] = (m + np.log(z))[:, 0]
        o[i] = np.einsum("ht,htd->hd", e / z, v[:, seen])
    return o, lse


def extend_chunked_expanded(q_nope, q_pe, w_uk, w_uv, kv_cache, block_row, seqlen, softmax_scale, chunk_tokens):
    """Extend of one request on the expanded path with its context in chunks: the T new
    tokens are the last T of the request's seqlen cached tokens (new token i at position
    seqlen - T + i, causal); the cached rows [c0, c0 + chunk_tokens) are expanded
    (expand_chunk), attended to (attend_chunk), and the chunks' (o, lse) merged by lse_merge.
    q_nope [T, H, 128], q_pe [T, H, 64] (RoPE already applied).  Returns o [T, H, 128], lse [T, H]."""
    q_nope = np.asarray(q_nope, dtype=np.float64)
    T = q_nope.shape[0]
    rows = gather_request(kv_cache, block_row, int(seqlen))
    qpos = np.arange(int(seqlen) - T, int(seqlen))
    parts_o, parts_l = [], []
    for c0 in range(0, int(seqlen), int(chunk_tokens)):
        c1 = min(int(seqlen), c0 + int(chunk_tokens))
        k_nope, k_pe, v = expand_chunk(rows[c0:c1], w_uk, w_uv)
        o, l = attend_chunk(q_nope, q_pe, k_nope, k_pe, v, np.arange(c0, c1), qpos, softmax_scale)
        parts_o.append(o)
        parts_l.append(l)
    return lse_merge(np.stack(parts_o), np.stack(parts_l))
