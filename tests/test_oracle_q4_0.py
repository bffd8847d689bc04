"""Pins of the oracle's q4_0 cache type (no GPU).

The pages name q4_0 as a llama.cpp KV type ("Sparse Attention -- Quest-style
block-selector ...", "All-KV-types composition") without defining it.
Reading R9: per group of 32 channels, m is the value of largest magnitude
(the first one in channel order), the f16 scale is d = fl16(fl32(m / -8)),
code = clamp(round-half-even(fl32(x / d)) + 8, 0, 15), value d * (code - 8);
byte i of a group holds channels 2i (low nibble) and 2i+1 (high nibble).

Pins: groups worked by hand; the quantizer against numpy float32/float16
arithmetic written independently here; the error bound; q4_0 attention
reducing to the q8_0 routine on the codes minus 8; the cache append.
"""
import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(404)


def _unpack(packed):
    packed = np.asarray(packed, np.uint8)
    out = np.empty(packed.size * 2, np.int64)
    out[0::2] = packed & 15
    out[1::2] = packed >> 4
    return out


@pytest.mark.parametrize("x,d,codes", [
    # m = 4: d = -0.5; 1 -> -2+8, -2 -> 4+8, 0.5 -> -1+8, 4 -> -8+8, zeros -> 8
    ([1.0, -2.0, 0.5, 4.0] + [0.0] * 28, -0.5, [6, 12, 7, 0] + [8] * 28),
    # a tie in magnitude: the first (-3) sets the sign, d = 0.375; 3 -> 8+8 clamps
    # to 15; 0.5625 / 0.375 = 1.5 -> 2 (half to even)
    ([-3.0, 3.0, 0.5625] + [0.0] * 29, 0.375, [0, 15, 10] + [8] * 29),
    # quotients on .5: 2.5 -> 2 and -1.5 -> -2 (half to even); m = -8: d = 1
    ([2.5, -1.5, -8.0, 3.5] + [0.0] * 28, 1.0, [10, 6, 0, 12] + [8] * 28),
    # an all-zero group: d = 0, every code 8
    ([0.0] * 32, 0.0, [8] * 32),
])
def test_q4_0_groups_worked_by_hand(x, d, codes):
    packed, dd = oracle.quantize_q4_0(np.array(x, np.float32))
    assert float(dd[0]) == d
    assert _unpack(packed).tolist() == codes


def _numpy_q4_0(x):
    x = np.asarray(x, np.float32).reshape(-1, 32)
    idx = np.argmax(np.abs(x), axis=1)           # first maximum in channel order
    m = x[np.arange(x.shape[0]), idx].astype(np.float64)
    d = (m / -8.0).astype(np.float32).astype(np.float16)
    df = d.astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        quot = np.where(df[:, None] != 0, x / df[:, None], np.float32(0))
    code = np.clip(np.rint(quot) + 8, 0, 15).astype(np.int64)
    return code.reshape(-1), d


@pytest.mark.parametrize("seed", range(6))
def test_q4_0_matches_numpy(seed):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal(128) * rng.choice([1e-5, 1e-2, 1.0, 20.0])).astype(np.float16)
    x = x.astype(np.float32)
    x[rng.integers(0, 128, 2)] *= -6.0
    packed, d = oracle.quantize_q4_0(x)
    want_code, want_d = _numpy_q4_0(x)
    assert np.array_equal(d.view(np.uint16), want_d.view(np.uint16))
    assert np.array_equal(_unpack(packed), want_code)


def test_q4_0_error_bound():
    x = (RNG.standard_normal(128 * 50) * 2.0).astype(np.float16).astype(np.float32)
    for r in range(50):
        row = x[r * 128:(r + 1) * 128]
        packed, d = oracle.quantize_q4_0(row)
        code = _unpack(packed)
        for g in range(4):
            dg = float(d[g])
            xg = row[g * 32:(g + 1) * 32].astype(np.float64)
            err = np.abs(xg - dg * (code[g * 32:(g + 1) * 32] - 8))
            # half a step; values of the other sign than m may clamp at +7 (one step)
            assert np.all(err <= abs(dg) * (1 + 1e-3) + 1e-12)
            j = np.argmax(np.abs(xg))
            assert code[g * 32 + j] in (0, 1)  # m itself lands on -8 (or -7 by f16 rounding)


def test_q4_0_attention_is_q8_0_on_codes_minus_8():
    L, D = 150, 128
    K4 = RNG.integers(0, 256, (L, D // 2)).astype(np.uint8)
    V4 = RNG.integers(0, 256, (L, D // 2)).astype(np.uint8)
    kd = RNG.uniform(-0.02, 0.02, (L, 4)).astype(np.float16)
    vd = RNG.uniform(-0.02, 0.02, (L, 4)).astype(np.float16)
    K8 = np.stack([_unpack(r) - 8 for r in K4]).astype(np.int8)
    V8 = np.stack([_unpack(r) - 8 for r in V4]).astype(np.int8)
    qc, qs = oracle.quantize_row(RNG.standard_normal(D).astype(np.float32))
    sel = np.array([0, 2], np.int32)
    for eps in (0.0, 0.7):
        got, dg = oracle.attend_q4_0(qc, qs, K4, V4, kd, vd, L, 64, 0.08, sel=sel, eps=eps)
        want, dw = oracle.attend_q8_0(qc, qs, K8, V8, kd, vd, L, 64, 0.08, sel=sel, eps=eps)
        assert dg == dw
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-15)


def test_q4_0_cache_append_matches_quantizer():
    B, Hkv, L = 1, 2, 70
    k = (RNG.standard_normal((B, L, Hkv, 128)) * 2).astype(np.float16)
    v = RNG.standard_normal((B, L, Hkv, 128)).astype(np.float16)
    oc = oracle.OracleCache(oracle.Q4_0, B, Hkv, 128, 128)
    oc.append(k[:, :40], v[:, :40])
    oc.append(k[:, 40:], v[:, 40:])
    for h in range(Hkv):
        for t in (0, 39, 40, 69):
            pk, dk = oracle.quantize_q4_0(k[0, t, h].astype(np.float32))
            assert np.array_equal(oc.K[0, h, t], pk)
            assert np.array_equal(oc.kd[0, h, t].view(np.uint16), dk.view(np.uint16))
            pv, dv = oracle.quantize_q4_0(v[0, t, h].astype(np.float32))
            assert np.array_equal(oc.V[0, h, t], pv)
            assert np.array_equal(oc.vd[0, h, t].view(np.uint16), dv.view(np.uint16))
    assert np.array_equal(oc.kmax[0, 1, 0], k[0, :64, 1].max(axis=0))
