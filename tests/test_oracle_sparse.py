"""Pins of the oracle's sparse (top-k) decode against facts other than itself:
the dense definition when every token is listed, dense attention over a cache
compacted to the listed tokens, pure-Python brute force, the closed form of a
single listed token, order invariance, causal masking and an empty list."""
import numpy as np

import oracle


def _case(rng, lens, B=None, s_q=1, H=3, extra=3):
    B = len(lens)
    nb = [(L + 63) // 64 for L in lens]
    pool = sum(nb) + extra
    perm = rng.permutation(pool)
    bt = np.full((B, max(nb)), -1, dtype=np.int64)
    pos = 0
    for b in range(B):
        bt[b, :nb[b]] = perm[pos:pos + nb[b]]
        pos += nb[b]
    kv = rng.standard_normal((pool, 64, 576))
    q = rng.standard_normal((B, s_q, H, 576))
    return q, kv, bt, np.array(lens)


def test_all_tokens_listed_equals_dense():
    rng = np.random.default_rng(20)
    q, kv, bt, lens = _case(rng, [70, 200, 1])
    idx = np.full((3, 200), -1)
    for b, L in enumerate(lens):
        idx[b, :L] = np.arange(L)
    for s_q, causal in ((1, False), (2, True)):
        qq = rng.standard_normal((3, s_q, 3, 576))
        o, l = oracle.decode_sparse(qq, kv, bt, lens, idx, lens, 0.05, causal=causal)
        od, ld = oracle.decode_absorbed(qq, kv, bt, lens, 0.05, causal=causal)
        assert np.allclose(o, od, rtol=0, atol=1e-12) and np.allclose(l, ld, rtol=0, atol=1e-12)


def test_equals_dense_over_a_compacted_cache():
    rng = np.random.default_rng(21)
    q, kv, bt, lens = _case(rng, [300, 129])
    k = [37, 100]
    idx = np.full((2, 100), -1)
    for b in range(2):
        idx[b, :k[b]] = rng.choice(lens[b], size=k[b], replace=False)
    o, l = oracle.decode_sparse(q, kv, bt, lens, idx, np.array(k), 0.07)
    for b in range(2):
        # the listed rows, in list order, as the pages of a new dense request
        t = idx[b, :k[b]]
        rows = kv[bt[b, t // 64], t % 64]
        pages = (k[b] + 63) // 64
        cache = np.zeros((pages, 64, 576))
        cache.reshape(-1, 576)[:k[b]] = rows
        od, ld = oracle.decode_absorbed(q[b:b + 1], cache, np.arange(pages)[None], np.array([k[b]]), 0.07)
        assert np.allclose(o[b], od[0], rtol=0, atol=1e-12) and np.allclose(l[b], ld[0], rtol=0, atol=1e-12)


def test_bruteforce_and_single_token_and_order():
    rng = np.random.default_rng(22)
    q, kv, bt, lens = _case(rng, [90])
    idx = np.array([[5, 80, 17, 64, 3, 88]])
    o, l = oracle.decode_sparse(q, kv, bt, lens, idx, np.array([6]), 0.1)
    keys = [kv[bt[0, t // 64], t % 64] for t in idx[0]]
    for h in range(3):
        ob, lb = oracle.decode_bruteforce(list(q[0, 0, h]), keys, 0.1)
        assert np.max(np.abs(np.array(ob) - o[0, 0, h])) < 1e-12 and abs(lb - l[0, 0, h]) < 1e-12
    # any order of the list gives the same result
    o2, l2 = oracle.decode_sparse(q, kv, bt, lens, idx[:, ::-1].copy(), np.array([6]), 0.1)
    assert np.allclose(o2, o, rtol=0, atol=1e-12) and np.allclose(l2, l, rtol=0, atol=1e-12)
    # a single listed token: out is its value, lse its scaled score
    o1, l1 = oracle.decode_sparse(q, kv, bt, lens, idx, np.array([1]), 0.1)
    row = kv[bt[0, 5 // 64], 5 % 64]
    assert np.allclose(o1[0, 0], row[:512][None], rtol=0, atol=1e-12)
    assert np.allclose(l1[0, 0], 0.1 * q[0, 0] @ row, rtol=0, atol=1e-12)


def test_causal_masks_listed_tokens_and_empty_list():
    rng = np.random.default_rng(23)
    q, kv, bt, lens = _case(rng, [50, 10], s_q=2)
    idx = np.array([[49, 10, 48], [0, -1, -1]])
    o, l = oracle.decode_sparse(q, kv, bt, lens, idx, np.array([3, 0]), 0.1, causal=True)
    # position 0 sees t <= 48 (drops 49); position 1 sees all three
    o0, l0 = oracle.decode_sparse(q[:1, :1], kv, bt[:1], lens[:1], np.array([[10, 48]]), np.array([2]), 0.1)
    assert np.allclose(o[0, 0], o0[0, 0], rtol=0, atol=1e-12) and np.allclose(l[0, 0], l0[0, 0], rtol=0, atol=1e-12)
    o1, l1 = oracle.decode_sparse(q[:1, 1:], kv, bt[:1], lens[:1], idx[:1], np.array([3]), 0.1)
    assert np.allclose(o[0, 1], o1[0, 0], rtol=0, atol=1e-12)
    # an empty list: out = 0, lse = -inf
    assert np.all(o[1] == 0) and np.all(np.isneginf(l[1]))
