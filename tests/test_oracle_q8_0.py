"""Pins of the oracle's q8_0 cache type (no GPU).

The pages name q8_0 as a llama.cpp KV type ("Sparse Attention -- Quest-style
block-selector ...", sections "All-KV-types composition" and "The decode win
lives on quantized KV") without defining it; reading R8 takes, per group of
32 channels, an f16 scale fl16(fl32(amax/127)) and codes round-half-even of
the f32 quotient x/d, clamped to +-127.

Pins: the oracle's binary16 rounding against numpy's conversion; the group
quantizer against numpy float32/float16 arithmetic written independently
here; its error bound and special cases; q8_0 attention reducing to the int8
attention routine when a row's group scales agree, and the uniform-logit
closed form.
"""
import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(808)


def test_half_rounding_matches_numpy():
    xs = np.concatenate([
        RNG.standard_normal(20000) * 10.0 ** RNG.integers(-9, 5, 20000),
        (np.arange(1, 3000) + 0.5) * 2.0 ** -24,              # subnormal ties
        (np.arange(1024, 2048) + 0.5) * 2.0 ** -10,           # normal ties in [1, 2)
        [0.0, -0.0, 65504.0, 65519.99, 65520.0, -65520.0, 6.1e-5, 6.09e-5],
    ])
    got = np.array([oracle.double_to_half(x) for x in xs], np.float16).view(np.uint16)
    with np.errstate(over="ignore"):
        want = xs.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want)


def _numpy_q8_0(x):
    x = np.asarray(x, np.float32).reshape(-1, 32)
    amax = np.abs(x).max(axis=1)
    s32 = (amax.astype(np.float64) / 127.0).astype(np.float32)
    d = s32.astype(np.float16)
    df = d.astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        quot = np.where(df[:, None] > 0, x / df[:, None], np.float32(0))
    code = np.clip(np.rint(quot), -127, 127).astype(np.int8)
    return code.reshape(-1), d


@pytest.mark.parametrize("seed", range(6))
def test_group_quantizer_matches_numpy(seed):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal(128) * rng.choice([1e-6, 1e-3, 1.0, 30.0])).astype(np.float16)
    x = x.astype(np.float32)
    x[rng.integers(0, 128, 3)] *= 8.0  # outlier channels in some groups
    code, d = oracle.quantize_group32(x)
    want_code, want_d = _numpy_q8_0(x)
    assert np.array_equal(d.view(np.uint16), want_d.view(np.uint16))
    assert np.array_equal(code, want_code)


def test_group_quantizer_bounds_and_special_cases():
    x = (RNG.standard_normal(128 * 64) * 3.0).astype(np.float16).astype(np.float32)
    for r in range(64):
        row = x[r * 128:(r + 1) * 128].copy()
        row[32:64] = 0.0                      # an all-zero group
        code, d = oracle.quantize_group32(row)
        df = d.astype(np.float64)
        assert df[1] == 0.0 and not code[32:64].any()
        assert np.abs(code.astype(np.int64)).max() <= 127
        for g in (0, 2, 3):
            xg = row[g * 32:(g + 1) * 32].astype(np.float64)
            err = np.abs(xg - df[g] * code[g * 32:(g + 1) * 32])
            # half a step, or the clamp at 127 steps when d rounded below amax/127
            lim = np.maximum(df[g] / 2, np.abs(xg) - 127 * df[g]) * (1 + 1e-6)
            assert np.all(err <= lim)
            # the largest magnitude lands within one code of +-127
            j = np.argmax(np.abs(xg))
            assert abs(int(code[g * 32 + j])) >= 126


def test_q8_0_equal_group_scales_reduce_to_int8():
    # when the four group scales of every row agree, the q8_0 logits and
    # values equal the int8 ones with that per-row scale
    L, D = 300, 128
    Kc = RNG.integers(-127, 128, (L, D)).astype(np.int8)
    Vc = RNG.integers(-127, 128, (L, D)).astype(np.int8)
    ks = RNG.uniform(0.001, 0.02, L).astype(np.float16)
    vs = RNG.uniform(0.001, 0.02, L).astype(np.float16)
    kd = np.repeat(ks[:, None], 4, axis=1)
    vd = np.repeat(vs[:, None], 4, axis=1)
    q = RNG.standard_normal(D).astype(np.float32)
    qc, qs = oracle.quantize_row(q)
    sel = np.array([0, 2, 3], np.int32)
    got, dropped = oracle.attend_q8_0(qc, qs, Kc, Vc, kd, vd, L, 64, 0.09, sel=sel)
    want = oracle.attend_int8(qc, qs, Kc, Vc, ks.astype(np.float32), vs.astype(np.float32),
                              L, 64, 0.09, sel=sel)
    assert dropped == 0.0
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-13)


def test_q8_0_group_scales_are_per_group():
    # token 0's key lives in group 2, token 1's in group 1, and the four key
    # scales of a row all differ: each logit carries its own group's scale,
    # so out = (w0 v0 + w1 v1) / (w0 + w1) with w = exp(logit) in closed form
    D = 128
    Kc = np.zeros((2, D), np.int8)
    Kc[0, 64:96] = 1
    Kc[1, 32:64] = 1
    Vc = np.ones((2, D), np.int8)
    qc = np.zeros(D, np.int8)
    qc[32:96] = 1
    kd = np.array([[1.0, 0.5, 0.03125, 2.0], [1.0, 0.0078125, 0.25, 2.0]], np.float16)
    vd = np.array([[1, 1, 1, 1], [2, 2, 2, 2]], np.float16)
    out, _ = oracle.attend_q8_0(qc, 1.0, Kc, Vc, kd, vd, 2, 64, 1.0)
    w0, w1 = np.exp(32 * 0.03125), np.exp(32 * 0.0078125)
    np.testing.assert_allclose(out, np.full(D, (w0 + 2 * w1) / (w0 + w1)), rtol=1e-14)


def test_q8_0_uniform_logits_closed_form():
    L, D = 130, 128
    Kc = RNG.integers(-127, 128, (L, D)).astype(np.int8)
    Vc = RNG.integers(-127, 128, (L, D)).astype(np.int8)
    kd = RNG.uniform(0.001, 0.02, (L, 4)).astype(np.float16)
    vd = RNG.uniform(0.001, 0.02, (L, 4)).astype(np.float16)
    qc = np.zeros(D, np.int8)
    out, _ = oracle.attend_q8_0(qc, 0.0, Kc, Vc, kd, vd, L, 64, 0.3)
    deq = Vc.astype(np.float64) * np.repeat(vd.astype(np.float64), 32, axis=1)
    np.testing.assert_allclose(out, deq.mean(axis=0), rtol=0, atol=1e-15)
    out, dropped = oracle.attend_q8_0(qc, 0.0, Kc, Vc, kd, vd, L, 64, 0.3, eps=1.5)
    assert dropped == 1.0 and not out.any()


def test_q8_0_cache_append_matches_group_quantizer():
    B, Hkv, L = 1, 2, 70
    k = (RNG.standard_normal((B, L, Hkv, 128)) * 2).astype(np.float16)
    v = RNG.standard_normal((B, L, Hkv, 128)).astype(np.float16)
    oc = oracle.OracleCache(oracle.Q8_0, B, Hkv, 128, 128)
    oc.append(k[:, :33], v[:, :33])
    oc.append(k[:, 33:], v[:, 33:])
    for h in range(Hkv):
        for t in (0, 32, 33, 69):
            code, d = oracle.quantize_group32(k[0, t, h].astype(np.float32))
            assert np.array_equal(oc.K[0, h, t], code)
            assert np.array_equal(oc.kd[0, h, t].view(np.uint16), d.view(np.uint16))
            code, d = oracle.quantize_group32(v[0, t, h].astype(np.float32))
            assert np.array_equal(oc.V[0, h, t], code)
            assert np.array_equal(oc.vd[0, h, t].view(np.uint16), d.view(np.uint16))
    # the bounds are the f16 keys' envelope, as for the other cache types
    assert np.array_equal(oc.kmax[0, 0, 0], k[0, :64, 0].max(axis=0))
    assert np.array_equal(oc.kmin[0, 1, 1], k[0, 64:70, 1].min(axis=0))
