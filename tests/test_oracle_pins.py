"""Pins of the CPU oracle against facts other than itself.

* the pages' tiny full-MLA example: absorbed and expanded paths agree and the
  cache holds 80 vs 20 numbers per token;
* brute force in pure Python on <= 8 tokens;
* closed forms: one token, zero query, identical values;
* a library routine: torch's scaled_dot_product_attention in float64 on CPU;
* the absorbed chain (absorb, decode, un-absorb) equals the expanded definition;
* the LSE merge of any KV split equals the unsplit result;
* RoPE: norm preservation, identity at position 0, relative-position property;
* planted mistakes (in the oracle, on the CPU) are caught by these pins.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import mla as om


def _rand_case(rng, B=2, s_q=1, H=4, lens=(5, 7), pool_extra=2, scale=0.1):
    nb = [(L + 63) // 64 for L in lens]
    pool = sum(nb) + pool_extra
    perm = rng.permutation(pool)
    bt = np.full((B, max(nb)), -1, dtype=np.int64)
    pos = 0
    for b in range(B):
        bt[b, :nb[b]] = perm[pos:pos + nb[b]]
        pos += nb[b]
    kv = rng.standard_normal((pool, 64, 576))
    q = rng.standard_normal((B, s_q, H, 576))
    return q, kv, bt, np.array(lens), scale


def test_tiny_full_mla_paths_agree():
    for seed in range(5):
        r = oracle.tiny_full_mla(seed)
        y1, y2 = r["y_expand"], r["y_absorb"]
        assert np.max(np.abs(y1 - y2)) <= 1e-10 * max(1.0, np.max(np.abs(y1)))
        assert np.max(np.abs(y1)) > 1e-3  # not trivially zero
    r = oracle.tiny_full_mla(0)
    assert r["cache_per_token_mha"] == 80 and r["cache_per_token_mla"] == 20


def test_bruteforce_small():
    rng = np.random.default_rng(1)
    q, kv, bt, lens, scale = _rand_case(rng, B=2, H=3, lens=(5, 8))
    out, lse = oracle.decode_absorbed(q, kv, bt, lens, scale)
    for b in range(2):
        keys = [kv[bt[b, t // 64], t % 64] for t in range(lens[b])]
        for h in range(3):
            o_bf, l_bf = oracle.decode_bruteforce(list(q[b, 0, h]), keys, scale)
            assert np.max(np.abs(np.array(o_bf) - out[b, 0, h])) < 1e-12
            assert abs(l_bf - lse[b, 0, h]) < 1e-12


def test_special_cases():
    rng = np.random.default_rng(2)
    q, kv, bt, _, scale = _rand_case(rng, B=1, H=2, lens=(1,))
    # one token: out is that token's latent, lse its score
    out, lse = oracle.decode_absorbed(q, kv, bt, np.array([1]), scale)
    row = kv[bt[0, 0], 0]
    assert np.array_equal(out[0, 0, 0], row[:512])
    assert abs(lse[0, 0, 1] - scale * float(q[0, 0, 1] @ row)) < 1e-12
    # zero query: uniform weights, out = mean of the values, lse = ln L
    L = 50
    q2, kv2, bt2, _, _ = _rand_case(rng, B=1, H=1, lens=(L,))
    q2[:] = 0
    out, lse = oracle.decode_absorbed(q2, kv2, bt2, np.array([L]), 0.3)
    vals = np.stack([kv2[bt2[0, t // 64], t % 64, :512] for t in range(L)])
    assert np.max(np.abs(out[0, 0, 0] - vals.mean(0))) < 1e-12
    assert abs(lse[0, 0, 0] - math.log(L)) < 1e-12
    # all values equal: the output is that value whatever the scores
    kv3 = kv2.copy()
    kv3[..., :512] = kv2[bt2[0, 0], 0, :512]
    q3 = rng.standard_normal(q2.shape)
    out, _ = oracle.decode_absorbed(q3, kv3, bt2, np.array([L]), 0.1)
    assert np.max(np.abs(out[0, 0, 0] - kv3[0, 0, :512])) < 1e-12
    # empty request and s_q > seqlen under causal masking: out = 0, lse = -inf
    out, lse = oracle.decode_absorbed(q3, kv3, bt2, np.array([0]), 0.1)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


@pytest.mark.parametrize("causal,s_q", [(False, 1), (False, 2), (True, 2), (True, 3)])
def test_against_sdpa_fp64(causal, s_q):
    """torch's attention routine on the contiguous (un-paged) tokens, float64."""
    rng = np.random.default_rng(3)
    lens = (70, 129)
    q, kv, bt, lens, scale = _rand_case(rng, B=2, s_q=s_q, H=5, lens=lens)
    out, lse = oracle.decode_absorbed(q, kv, bt, lens, scale, causal=causal)
    for b in range(2):
        L = lens[b]
        keys = np.stack([kv[bt[b, t // 64], t % 64] for t in range(L)])
        K = torch.tensor(keys)[None, None].expand(1, 5, L, 576)
        V = torch.tensor(keys[:, :512])[None, None].expand(1, 5, L, 512)
        Q = torch.tensor(q[b]).permute(1, 0, 2)[None]          # [1, H, s_q, 576]
        mask = None
        if causal:
            t = torch.arange(L)[None, :]
            i = torch.arange(s_q)[:, None]
            mask = t <= (L - s_q + i)                              # bottom-right aligned
        ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=scale)
        ref = ref[0].permute(1, 0, 2).numpy()                      # [s_q, H, 512]
        assert np.max(np.abs(ref - out[b])) < 1e-12
        # lse from torch's logsumexp on the masked scores
        S = scale * torch.einsum("hid,htd->hit", Q[0], K[0])
        if mask is not None:
            S = S.masked_fill(~mask, float("-inf"))
        ref_lse = torch.logsumexp(S, -1).permute(1, 0).numpy()
        assert np.max(np.abs(ref_lse - lse[b])) < 1e-12


def test_weighted_magnitude_output():
    rng = np.random.default_rng(9)
    q, kv, bt, lens, scale = _rand_case(rng, B=2, H=3, lens=(70, 129))
    out, lse, out_abs = oracle.decode_absorbed(q, kv, bt, lens, scale, with_abs=True)
    assert np.all(np.abs(out) <= out_abs + 1e-12)                  # triangle inequality
    o2, l2 = oracle.decode_absorbed(q, np.abs(kv), bt, lens, scale)  # with |v| as values
    # same scores only where the key part is unchanged: compare on a case with non-negative cache
    kvp = np.abs(kv)
    out_p, _, abs_p = oracle.decode_absorbed(q, kvp, bt, lens, scale, with_abs=True)
    assert np.max(np.abs(out_p - abs_p)) < 1e-12                    # non-negative values: equal


def test_causal_alignment_matches_shorter_context():
    rng = np.random.default_rng(4)
    q, kv, bt, lens, scale = _rand_case(rng, B=1, s_q=2, H=3, lens=(100,))
    out, lse = oracle.decode_absorbed(q, kv, bt, lens, scale, causal=True)
    # position 0 (earliest new token) sees 99 tokens, position 1 sees all 100
    o0, l0 = oracle.decode_absorbed(q[:, :1], kv, bt, np.array([99]), scale)
    o1, l1 = oracle.decode_absorbed(q[:, 1:], kv, bt, np.array([100]), scale)
    assert np.array_equal(out[:, 0], o0[:, 0]) and np.array_equal(lse[:, 0], l0[:, 0])
    assert np.array_equal(out[:, 1], o1[:, 0]) and np.array_equal(lse[:, 1], l1[:, 0])


def test_paging_is_only_indexing():
    """The same logical tokens under another page permutation give the same result."""
    rng = np.random.default_rng(5)
    q, kv, bt, lens, scale = _rand_case(rng, B=2, H=4, lens=(130, 200), pool_extra=3)
    out, lse = oracle.decode_absorbed(q, kv, bt, lens, scale)
    perm = rng.permutation(kv.shape[0])
    inv = np.argsort(perm)
    kv2 = kv[perm]                 # page p of kv2 holds page perm[p] of kv
    bt2 = np.where(bt >= 0, inv[np.maximum(bt, 0)], -1)
    out2, lse2 = oracle.decode_absorbed(q, kv2, bt2, lens, scale)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


@pytest.mark.parametrize("causal,s_q", [(False, 1), (True, 2)])
def test_absorbed_chain_equals_expanded(causal, s_q):
    rng = np.random.default_rng(6)
    B, H = 2, 6
    lens = np.array([77, 140])
    q, kv, bt, lens, _ = _rand_case(rng, B=B, s_q=s_q, H=H, lens=tuple(lens))
    q_nope = rng.standard_normal((B, s_q, H, 128))
    q_pe = rng.standard_normal((B, s_q, H, 64))
    w_uk = rng.standard_normal((H, 128, 512)) / math.sqrt(512)
    w_uv = rng.standard_normal((H, 512, 128)) / math.sqrt(512)
    scale = 1 / math.sqrt(192)
    q_lat = oracle.absorb_q(q_nope.reshape(B * s_q, H, 128), w_uk).reshape(B, s_q, H, 512)
    qq = np.concatenate([q_lat, q_pe], axis=-1)
    o_lat, lse_a = oracle.decode_absorbed(qq, kv, bt, lens, scale, causal=causal)
    o_abs = oracle.unabsorb_o(o_lat.reshape(B * s_q, H, 512), w_uv).reshape(B, s_q, H, 128)
    o_exp, lse_e = oracle.decode_expanded(q_nope, q_pe, w_uk, w_uv, kv, bt, lens, scale, causal=causal)
    assert np.max(np.abs(o_abs - o_exp)) < 1e-10
    assert np.max(np.abs(lse_a - lse_e)) < 1e-10
    assert np.max(np.abs(o_exp)) > 1e-3


def test_lse_merge_of_any_split_equals_unsplit():
    rng = np.random.default_rng(7)
    q, kv, bt, lens, scale = _rand_case(rng, B=1, H=4, lens=(300,))
    L = 300
    keys = np.stack([kv[bt[0, t // 64], t % 64] for t in range(L)])
    full_o, full_l = oracle.decode_absorbed(q, kv, bt, lens, scale)
    for trial in range(10):
        k = rng.integers(1, 7)
        cuts = np.sort(rng.choice(np.arange(1, L), size=k - 1, replace=False)) if k > 1 else []
        edges = [0, *cuts, L]
        os_, ls_ = [], []
        for a, b in zip(edges[:-1], edges[1:]):
            kv_seg = keys[a:b][None]                              # one page-free "block"
            # lay the segment out as its own paged cache
            n = b - a
            nbk = (n + 63) // 64
            pages = np.zeros((nbk, 64, 576))
            pages.reshape(-1, 576)[:n] = kv_seg[0]
            o, l_ = oracle.decode_absorbed(q, pages, np.arange(nbk)[None], np.array([n]), scale)
            os_.append(o)
            ls_.append(l_)
        # an empty part carries no weight
        os_.append(np.full_like(os_[0], 123.0))
        ls_.append(np.full_like(ls_[0], -np.inf))
        mo, ml = oracle.lse_merge(np.stack(os_), np.stack(ls_))
        assert np.max(np.abs(mo - full_o)) < 1e-12
        assert np.max(np.abs(ml - full_l)) < 1e-12
    mo, ml = oracle.lse_merge(np.ones((2, 3, 4)), np.full((2, 3), -np.inf))
    assert np.all(mo == 0) and np.all(np.isneginf(ml))


def test_rope_properties():
    rng = np.random.default_rng(8)
    T, R = 9, 8
    x = rng.standard_normal((T, R))
    y = om.rope_interleaved(x, np.arange(T))
    assert np.allclose(y[0], x[0], atol=0, rtol=0)                       # position 0: identity
    n_x = x[:, 0::2] ** 2 + x[:, 1::2] ** 2
    n_y = y[:, 0::2] ** 2 + y[:, 1::2] ** 2
    assert np.max(np.abs(n_x - n_y)) < 1e-12                              # pairs keep their norm
    # <rope(a, m), rope(b, n)> depends only on m - n
    a, b = rng.standard_normal(R), rng.standard_normal(R)
    def dot(m, n):
        ra = om.rope_interleaved(np.tile(a, (max(m, n) + 1, 1)), np.arange(max(m, n) + 1))[m]
        rb = om.rope_interleaved(np.tile(b, (max(m, n) + 1, 1)), np.arange(max(m, n) + 1))[n]
        return ra @ rb
    assert abs(dot(5, 2) - dot(7, 4)) < 1e-12 and abs(dot(3, 3) - a @ b) < 1e-12
    # first pair rotates by exactly pos radians (base^0 = 1)
    e = np.zeros((3, R)); e[:, 0] = 1.0
    r = om.rope_interleaved(e, np.arange(3))
    assert abs(r[2, 0] - math.cos(2.0)) < 1e-15 and abs(r[2, 1] - math.sin(2.0)) < 1e-15


def test_assemble_q_layout_and_rope_per_token():
    rng = np.random.default_rng(12)
    N, H = 5, 3
    q_nope = rng.standard_normal((N, H, 128))
    w_uk = rng.standard_normal((H, 128, 512)) / math.sqrt(512)
    q_pe = rng.standard_normal((N, H, 64))
    plain = om.assemble_q(q_nope, q_pe, w_uk)
    assert plain.shape == (N, H, 576)
    assert np.array_equal(plain[..., 512:], q_pe)
    assert np.allclose(plain[..., :512], np.einsum("nhd,hdc->nhc", q_nope, w_uk), rtol=0, atol=1e-12)
    assert np.array_equal(om.assemble_q(q_nope, q_pe, w_uk, positions=np.zeros(N)), plain)   # pos 0: identity
    # every token turns by its own position: a unit vector in dim 0 ends at (cos p, sin p);
    # in the last pair (j = 31) the angle is p * base^(-62/64)
    pos = np.array([0, 1, 7, 4096, 131071])
    e0 = np.zeros((N, H, 64)); e0[..., 0] = 1.0
    e62 = np.zeros((N, H, 64)); e62[..., 62] = 1.0
    r0 = om.assemble_q(q_nope, e0, w_uk, positions=pos)[..., 512:]
    r62 = om.assemble_q(q_nope, e62, w_uk, positions=pos)[..., 512:]
    for n, p in enumerate(pos):
        assert np.allclose(r0[n, :, 0], math.cos(p), atol=1e-12) and np.allclose(r0[n, :, 1], math.sin(p), atol=1e-12)
        a = p * 10000.0 ** (-62.0 / 64.0)
        assert np.allclose(r62[n, :, 62], math.cos(a), atol=1e-12)
        assert np.allclose(r62[n, :, 63], math.sin(a), atol=1e-12)
    rot = om.assemble_q(q_nope, q_pe, w_uk, positions=pos)[..., 512:]
    assert np.allclose(rot[..., 0::2] ** 2 + rot[..., 1::2] ** 2, q_pe[..., 0::2] ** 2 + q_pe[..., 1::2] ** 2,
                       atol=1e-12)


# ---- planted mistakes: each must make at least one pin fail -----------------------------

def _pins_pass():
    try:
        test_bruteforce_small()
        test_special_cases()
        test_against_sdpa_fp64(False, 1)
        test_against_sdpa_fp64(True, 2)
        test_absorbed_chain_equals_expanded(False, 1)
        return True
    except (AssertionError, ValueError, IndexError):
        return False


def test_pins_catch_planted_mistakes(monkeypatch):
    assert _pins_pass()
    real_gather = om.gather_request
    real_vis = om.visible_tokens

    mutants = {
        "drop the last token": lambda m: m.setattr(om, "gather_request",
            lambda kv, row, n, sc=None: np.concatenate([real_gather(kv, row, n, sc)[:-1],
                                                       real_gather(kv, row, n, sc)[:1] * 0], 0)),
        "shift one page": lambda m: m.setattr(om, "gather_request",
            lambda kv, row, n, sc=None: real_gather(kv, np.roll(np.asarray(row), 1), n, sc)),
        "causal off by one": lambda m: m.setattr(om, "visible_tokens",
            lambda L, s_q, i, c: max(0, real_vis(L, s_q, i, c) - (1 if c else 0))),
        "value includes rope dims": lambda m: m.setattr(om, "D_LATENT", 511),
    }
    for name, plant in mutants.items():
        with monkeypatch.context() as m:
            plant(m)
            assert not _pins_pass(), f"planted mistake not caught: {name}"
    assert _pins_pass()
