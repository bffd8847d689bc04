"""Pins of the oracle's f32-input append (no GPU).

"cpu-attn" (Usage): the cache takes each token's K and V as f32.  "Sparse
Attention -- Quest-style block-selector ...", "All-KV-types composition": the
bounds come from the keys before quantization.  Reading R11: the f16 cache
stores each value's nearest f16; the quantized caches quantize the f32 values
and round the f32 keys' block envelope outward to f16.

Pins: directed binary16 rounding against numpy's float16 conversion and
nextafter; the f16 cache against the f16-input append of numpy-rounded values;
the quantized rows against the row quantizers on the f32 values; the bounds as
the tightest f16 pair that still holds every f32 key, across chunked appends.
"""
import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(3232)


def _numpy_dir(x, direction):
    with np.errstate(over="ignore"):
        h = np.float16(x)
        if direction < 0 and float(h) > x:
            h = np.nextafter(h, np.float16(-np.inf))
        if direction > 0 and float(h) < x:
            h = np.nextafter(h, np.float16(np.inf))
    return h


def test_directed_rounding_matches_numpy():
    xs = np.concatenate([
        RNG.standard_normal(5000) * 10.0 ** RNG.integers(-8, 5, 5000),
        (np.arange(1, 500) + 0.25) * 2.0 ** -24,                # subnormals off the grid
        [0.0, -0.0, 2.0 ** -25, -(2.0 ** -25), 65504.0, 65519.0, 65520.0, 70000.0, -70000.0,
         1.0, -1.0, 1.0 + 2 ** -12, -(1.0 + 2 ** -12)],
    ])
    for x in xs:
        for direction in (-1, 1):
            got = oracle.double_to_half_dir(x, direction)
            want = _numpy_dir(x, direction)
            assert got.view(np.uint16) == want.view(np.uint16) or (got == want == 0), \
                (x, direction, got, want)
            # and it lies on the asked side of x
            assert (float(got) <= x) if direction < 0 else (float(got) >= x)


def _inputs(B, L, Hkv, scale=2.0, seed=0):
    rng = np.random.default_rng(seed)
    k = (rng.standard_normal((B, L, Hkv, 128)) * scale).astype(np.float32)
    v = rng.standard_normal((B, L, Hkv, 128)).astype(np.float32)
    k[0, :3, 0, :4] = [[1e-6, -1e-6, 3e4, -3e4]] * 3   # subnormal and large keys
    return k, v


def test_f16_cache_stores_the_nearest_f16():
    B, L, Hkv = 2, 150, 3
    k, v = _inputs(B, L, Hkv)
    a = oracle.OracleCache(oracle.F16, B, Hkv, 128, 256)
    a.append_f32(k[:, :70], v[:, :70])
    a.append_f32(k[:, 70:], v[:, 70:])
    b = oracle.OracleCache(oracle.F16, B, Hkv, 128, 256)
    b.append(k.astype(np.float16), v.astype(np.float16))   # numpy's own rounding
    assert np.array_equal(a.K.view(np.uint16), b.K.view(np.uint16))
    assert np.array_equal(a.V.view(np.uint16), b.V.view(np.uint16))
    assert np.array_equal(a.kmin.view(np.uint16), b.kmin.view(np.uint16))
    assert np.array_equal(a.kmax.view(np.uint16), b.kmax.view(np.uint16))


@pytest.mark.parametrize("dtype", [oracle.INT8, oracle.Q8_0, oracle.Q4_0])
def test_quantized_rows_come_from_the_f32_values(dtype):
    B, L, Hkv = 1, 70, 2
    k, v = _inputs(B, L, Hkv, seed=dtype)
    oc = oracle.OracleCache(dtype, B, Hkv, 128, 128)
    oc.append_f32(k, v)
    quant = {oracle.INT8: oracle.quantize_row, oracle.Q8_0: oracle.quantize_group32,
             oracle.Q4_0: oracle.quantize_q4_0}[dtype]
    for h in range(Hkv):
        for t in (0, 1, 33, 69):
            for x, rows, scl in ((k, oc.K, oc.ks if dtype == oracle.INT8 else oc.kd),
                                 (v, oc.V, oc.vs if dtype == oracle.INT8 else oc.vd)):
                code, s = quant(x[0, t, h])
                assert np.array_equal(rows[0, h, t], code)
                want = np.atleast_1d(np.asarray(s, scl.dtype)).tobytes()
                assert np.atleast_1d(scl[0, h, t]).tobytes() == want


@pytest.mark.parametrize("dtype", [oracle.INT8, oracle.Q8_0, oracle.Q4_0])
@pytest.mark.parametrize("chunks", [[200], [1] * 5 + [60, 70, 65], [64, 64, 72]])
def test_bounds_are_the_tightest_outward_f16_pair(dtype, chunks):
    B, Hkv, L = 1, 2, sum(chunks)
    k, v = _inputs(B, L, Hkv, scale=3.0, seed=len(chunks))
    oc = oracle.OracleCache(dtype, B, Hkv, 128, 256)
    s = 0
    for n in chunks:
        oc.append_f32(k[:, s:s + n], v[:, s:s + n])
        s += n
    for h in range(Hkv):
        for j in range((L + 63) // 64):
            blk = k[0, j * 64:min(L, j * 64 + 64), h].astype(np.float64)
            lo, hi = blk.min(axis=0), blk.max(axis=0)
            kmin = oc.kmin[0, h, j].astype(np.float64)
            kmax = oc.kmax[0, h, j].astype(np.float64)
            assert np.all(kmin <= lo) and np.all(kmax >= hi)          # they bound every key
            up = np.nextafter(oc.kmin[0, h, j], np.float16(np.inf)).astype(np.float64)
            dn = np.nextafter(oc.kmax[0, h, j], np.float16(-np.inf)).astype(np.float64)
            assert np.all(up > lo) and np.all(dn < hi)                # and none is looser
