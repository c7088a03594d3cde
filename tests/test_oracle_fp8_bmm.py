"""Pins of the oracle's FP8 projections (input_to_float8 + bmm_fp8) against the E4M3
format, a library conversion, exact integer arithmetic, pure-Python brute force and the
(separately pinned) bf16 absorption; planted mistakes must fail one of them."""
import fractions

import numpy as np
import pytest
import torch

import oracle
import oracle.mla as om


def _rounding_agrees_with_torch(n=20000, seed=0):
    rng = np.random.default_rng(seed)
    mag = np.exp2(rng.uniform(-14, np.log2(460.0), size=n)).astype(np.float32)
    v = mag * rng.choice([-1.0, 1.0], size=n).astype(np.float32)
    # exact midpoints between neighbouring codes are the ties the rounding must send to even
    pos = oracle.E4M3_VALUES[1:126]
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    v = np.concatenate([v, mids, -mids, np.float32([0.0, -0.0, 2.0 ** -10, -2.0 ** -10, 448.0, -448.0])])
    ours = om.e4m3_round(v)
    lib = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return np.array_equal(ours, lib)


def test_e4m3_round_matches_library_conversion_in_range():
    assert _rounding_agrees_with_torch()


def test_e4m3_round_saturates_and_round_trips():
    big = np.array([448.0, 449.0, 464.0, 465.0, 1e6, np.inf, -500.0, -np.inf])
    assert om.e4m3_round(big).tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]
    assert om.e4m3_round(np.array([np.nan])).tolist() == [0x7F]
    finite = [c for c in range(256) if c not in (0x7F, 0xFF)]
    assert np.array_equal(om.e4m3_round(oracle.E4M3_VALUES[finite]), np.array(finite, dtype=np.uint8))


def _quantization_ok(x):
    codes, scale = oracle.input_to_float8(x)
    xv = np.asarray(x, dtype=np.float64)
    deq = oracle.E4M3_VALUES[codes] * scale
    amax = np.abs(xv).max()
    if amax == 0:
        return scale == 1.0 and not codes.any() & 0x7F
    k = np.unravel_index(np.argmax(np.abs(xv)), xv.shape)
    if abs(abs(oracle.E4M3_VALUES[codes[k]]) - 448.0) > 0:      # the largest magnitude lands on 448
        return False
    if abs(scale - amax / 448.0) > 1e-6 * scale:                 # scale = amax / 448
        return False
    normal = np.abs(xv) >= 2.0 ** -6 * scale
    rel = np.abs(deq - xv)[normal] / np.abs(xv)[normal]
    sub_err = np.abs(deq - xv)[~normal]
    return bool(np.all(np.isfinite(deq)) and rel.max(initial=0) <= 2.0 ** -4 + 1e-6
                and sub_err.max(initial=0) <= 2.0 ** -10 * scale * (1 + 1e-6))


def test_input_to_float8_maps_the_extreme_to_448_within_half_a_step():
    rng = np.random.default_rng(1)
    for shape, sd in (((5, 3, 128), 1.0), ((2, 4, 512), 1e-3), ((1, 1, 128), 40.0)):
        x = torch.from_numpy(rng.standard_normal(shape) * sd).to(torch.bfloat16).float().numpy()
        assert _quantization_ok(x)
    z = np.zeros((2, 2, 128))
    codes, scale = oracle.input_to_float8(z)
    assert scale == 1.0 and np.all(oracle.E4M3_VALUES[codes] == 0)
    # a power-of-two rescaling of the input keeps the codes and rescales the scale
    x = torch.from_numpy(rng.standard_normal((3, 2, 128))).to(torch.bfloat16).float().numpy()
    c1, s1 = oracle.input_to_float8(x)
    c2, s2 = oracle.input_to_float8(x * 8.0)
    assert np.array_equal(c1, c2) and s2 == 8.0 * s1


def test_bmm_fp8_brute_force_and_exact_integers():
    rng = np.random.default_rng(2)
    N, H, J, K = 3, 2, 5, 64
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    x = rng.choice(finite, size=(N, H, K))
    w = rng.choice(finite, size=(H, J, K))
    xs, ws = 0.75, 2.0 ** -9
    y = oracle.bmm_fp8(x, xs, w, ws)
    for n in range(N):                                           # exact rational arithmetic
        for h in range(H):
            for j in range(J):
                acc = fractions.Fraction(0)
                for k in range(K):
                    acc += fractions.Fraction(oracle.E4M3_VALUES[x[n, h, k]]) * fractions.Fraction(oracle.E4M3_VALUES[w[h, j, k]])
                ref = float(acc * fractions.Fraction(xs) * fractions.Fraction(ws))
                assert abs(y[n, h, j] - ref) <= 1e-12 * max(1.0, abs(ref))
    # small integers are exact in E4M3: the product is an integer matmul times the scales
    ints = np.arange(-8, 9)
    xi = rng.choice(ints, size=(N, H, K))
    wi = rng.choice(ints, size=(H, J, K))
    y2 = oracle.bmm_fp8(om.e4m3_round(xi), 0.5, om.e4m3_round(wi), 0.25)
    ref2 = np.einsum("nhk,hjk->nhj", xi.astype(np.int64), wi.astype(np.int64)) * 0.125
    assert np.array_equal(y2, ref2)


def test_fp8_absorption_is_the_bf16_absorption_of_the_decoded_operands():
    # W_UK[h] is [128, 512]; the FP8 weight is stored transposed, [512, 128] per head
    rng = np.random.default_rng(3)
    N, H = 6, 3
    q_nope = torch.from_numpy(rng.standard_normal((N, H, 128))).to(torch.bfloat16).float().numpy()
    w = rng.standard_normal((H, 128, 512)) / np.sqrt(512)
    w_scale = 2.0 ** -9
    w_t = om.e4m3_round(np.transpose(w, (0, 2, 1)) / w_scale)
    got = oracle.absorb_q_fp8(q_nope, w_t, w_scale)
    codes, xs = oracle.input_to_float8(q_nope)
    w_dec = np.transpose(oracle.E4M3_VALUES[w_t], (0, 2, 1)) * w_scale
    ref = oracle.absorb_q(oracle.E4M3_VALUES[codes] * xs, w_dec)
    assert np.max(np.abs(got - ref)) <= 1e-12 * np.max(np.abs(ref))
    # and it approximates the exact bf16 product to FP8 accuracy
    exact = oracle.absorb_q(q_nope, w)
    assert np.linalg.norm(got - exact) / np.linalg.norm(exact) < 0.05
    o_lat = torch.from_numpy(rng.standard_normal((N, H, 512))).to(torch.bfloat16).float().numpy()
    wv = rng.standard_normal((H, 512, 128)) / np.sqrt(512)
    wv_t = om.e4m3_round(np.transpose(wv, (0, 2, 1)) / w_scale)
    got_o = oracle.unabsorb_o_fp8(o_lat, wv_t, w_scale)
    c_o, s_o = oracle.input_to_float8(o_lat)
    ref_o = oracle.unabsorb_o(oracle.E4M3_VALUES[c_o] * s_o, np.transpose(oracle.E4M3_VALUES[wv_t], (0, 2, 1)) * w_scale)
    assert np.max(np.abs(got_o - ref_o)) <= 1e-12 * np.max(np.abs(ref_o))


def _all_pins_pass():
    try:
        assert _rounding_agrees_with_torch(3000)
        test_e4m3_round_saturates_and_round_trips()
        test_input_to_float8_maps_the_extreme_to_448_within_half_a_step()
        test_bmm_fp8_brute_force_and_exact_integers()
        test_fp8_absorption_is_the_bf16_absorption_of_the_decoded_operands()
    except AssertionError:
        return False
    return True


def test_pins_catch_planted_mistakes(monkeypatch):
    assert _all_pins_pass()
    real_round, real_bmm, real_q = om.e4m3_round, om.bmm_fp8, om.input_to_float8

    def round_half_up(v):   # ties away from zero instead of to even
        v = np.asarray(v, dtype=np.float64)
        return real_round(v + np.sign(v) * np.abs(v) * 1e-9)

    def scale_inverted(x):  # the reciprocal scale returned
        c, s = real_q(x)
        return c, 1.0 / s

    mutants = {
        "ties rounded away from zero": lambda m: m.setattr(om, "e4m3_round", round_half_up),
        "weight rows shifted by one": lambda m: m.setattr(om, "bmm_fp8",
            lambda x, xs, w, ws: real_bmm(x, xs, np.roll(w, 1, axis=1), ws)),
        "input scale inverted": lambda m: m.setattr(om, "input_to_float8", scale_inverted),
    }
    for name, plant in mutants.items():
        with monkeypatch.context() as m:
            plant(m)
            assert not _all_pins_pass(), f"planted mistake not caught: {name}"
    assert _all_pins_pass()
