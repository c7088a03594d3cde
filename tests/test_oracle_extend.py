"""Pins of the oracle's chunked expanded extend (MHA_CHUNKED_KV): chunked and merged by LSE
it must equal the unchunked expanded definition and the absorbed chain (the pages' two
equivalent paths), for every chunk size; planted mistakes must fail those pins."""
import numpy as np
import pytest

import oracle
import oracle.mla as om


def _case(seed=0, T=5, L=300, H=3):
    rng = np.random.default_rng(seed)
    nb = (L + 63) // 64
    pool = nb + 3
    bt = rng.permutation(pool)[:nb]
    kv = rng.standard_normal((pool, 64, 576))
    q_nope = rng.standard_normal((T, H, 128))
    q_pe = rng.standard_normal((T, H, 64))
    w_uk = rng.standard_normal((H, 128, 512)) / np.sqrt(512)
    w_uv = rng.standard_normal((H, 512, 128)) / np.sqrt(512)
    return q_nope, q_pe, w_uk, w_uv, kv, bt, L, 1.0 / np.sqrt(192.0)


def _pins_hold():
    q_nope, q_pe, w_uk, w_uv, kv, bt, L, scale = _case()
    T = q_nope.shape[0]
    ref_o, ref_l = oracle.decode_expanded(q_nope[None], q_pe[None], w_uk, w_uv, kv, bt[None], np.array([L]), scale,
                                          causal=True)
    q = np.concatenate([oracle.absorb_q(q_nope, w_uk), q_pe], axis=-1)[None]
    lat, lat_l = oracle.decode_absorbed(q, kv, bt[None], np.array([L]), scale, causal=True)
    abs_o = oracle.unabsorb_o(lat[0], w_uv)
    for chunk in (1, 64, 100, 256, L):
        o, l = oracle.extend_chunked_expanded(q_nope, q_pe, w_uk, w_uv, kv, bt, L, scale, chunk)
        if not (np.allclose(o, ref_o[0], atol=1e-10, rtol=1e-10) and np.allclose(l, ref_l[0], atol=1e-10, rtol=0)):
            return False
        if not (np.allclose(o, abs_o, atol=1e-9, rtol=1e-9) and np.allclose(l, lat_l[0], atol=1e-9, rtol=0)):
            return False
    return T == 5


def test_chunked_extend_equals_unchunked_and_absorbed_paths():
    assert _pins_hold()


def test_expand_chunk_shapes_and_rope_key_shared():
    q_nope, q_pe, w_uk, w_uv, kv, bt, L, scale = _case(1, L=70)
    rows = oracle.gather_request(kv, bt, L)
    k_nope, k_pe, v = oracle.expand_chunk(rows, w_uk, w_uv)
    assert k_nope.shape == (3, 70, 128) and k_pe.shape == (70, 64) and v.shape == (3, 70, 128)
    assert np.array_equal(k_pe, rows[:, 512:])
    # one head and one token by hand: k = W_UK[h] c, v = W_UV[h]^T c
    assert np.allclose(k_nope[2, 5], w_uk[2] @ rows[5, :512])
    assert np.allclose(v[1, 7], rows[7, :512] @ w_uv[1])


def test_queries_before_a_chunk_see_nothing_of_it():
    q_nope, q_pe, w_uk, w_uv, kv, bt, L, scale = _case(2, T=4, L=130)
    rows = oracle.gather_request(kv, bt, L)
    k_nope, k_pe, v = oracle.expand_chunk(rows[128:130], w_uk, w_uv)
    qpos = np.arange(L - 4, L)                      # 126..129
    o, l = oracle.attend_chunk(q_nope, q_pe, k_nope, k_pe, v, np.arange(128, 130), qpos, scale)
    assert np.all(np.isneginf(l[:2])) and np.all(o[:2] == 0)     # positions 126, 127
    assert np.all(np.isfinite(l[2:]))


def test_pins_catch_planted_mistakes(monkeypatch):
    assert _pins_hold()
    real_attend, real_expand, real_merge = om.attend_chunk, om.expand_chunk, om.lse_merge
    mutants = {
        "chunks averaged instead of merged by lse": lambda m: m.setattr(om, "lse_merge",
            lambda o, l: (np.mean(np.asarray(o), axis=0), np.max(np.asarray(l), axis=0))),
        "causal limit off by one": lambda m: m.setattr(om, "attend_chunk",
            lambda qn, qp, kn, kp, v, kpos, qpos, sc: real_attend(qn, qp, kn, kp, v, kpos, np.asarray(qpos) - 1, sc)),
        "value expanded with the wrong head": lambda m: m.setattr(om, "expand_chunk",
            lambda rows, wk, wv: (lambda k, p, v: (k, p, np.roll(v, 1, axis=0)))(*real_expand(rows, wk, wv))),
    }
    for name, plant in mutants.items():
        with monkeypatch.context() as m:
            plant(m)
            assert not _pins_hold(), f"planted mistake not caught: {name}"
    assert _pins_hold()


def test_output_allowance_covers_score_moves():
    # the parity harness's expanded-path output allowance: if every score of a row moves by at
    # most d, an attention output moves by at most (e^2d - 1) * sum_t p_t |v_t|; checked on
    # random rows and values with random moves inside d, including moves of +d / -d on
    # different keys (the worst case)
    import sys, os
    sys.path.insert(0, os.path.dirname(__file__))
    from _harness import expanded_output_allowance
    rng = np.random.default_rng(3)
    for trial in range(200):
        n = int(rng.integers(1, 50))
        s = rng.normal(0, 3, n)
        v = rng.normal(0, 2, (n, 4))
        d = float(rng.uniform(0, 0.3))
        ds = rng.choice([-d, d], n) if trial % 2 else rng.uniform(-d, d, n)
        p = np.exp(s - s.max()); p /= p.sum()
        p2 = np.exp(s + ds - (s + ds).max()); p2 /= p2.sum()
        moved = np.abs(p2 @ v - p @ v)
        bound = expanded_output_allowance(np.array([[d]]), (p @ np.abs(v))[None, None, :])[0, 0]
        assert np.all(moved <= bound * (1 + 1e-12) + 1e-15), (trial, moved, bound)
