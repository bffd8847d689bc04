"""Pins of the oracle's moment tail to facts outside itself (no GPU).

"SCSA: Self-Calibrating Subquadratic Attention", section "2. Mechanism":
every group of keys that is not read exactly contributes its member count m
times exp(a), a = scale * q . c_K, at its value mean c_V, inside the shared
softmax normalizer; the output is (exact numerator + tail numerator) /
(exact mass + tail mass).  Reading R10 applies it to the Quest blocks the
selection leaves out, with c_K, c_V the f16-rounded means of the block's
stored (dequantized) rows and q the unquantized query.

Pins: hand-worked cases (tests/golden/moment_tail.txt); the block means
against numpy's own mean and float16 conversion; the exact part against the
per-type attention functions already pinned (every block listed); blocks of
equal keys, where the tail is exact, against dense attention; q = 0, where
every weight is a count, against the plain mean of the values.
"""
import math
import os

import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(1010)
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "moment_tail.txt")
R3 = 0.333251953125  # the binary16 nearest to 1/3


def _term(s):
    total = 0.0
    for piece in s.split("+"):
        if piece.startswith("ln"):
            total += math.log(float(piece[2:]))
        elif piece.endswith("r3"):
            total += (float(piece[:-3]) if piece != "r3" else 1.0) * R3
        else:
            total += float(piece)
    return total


def _rows(s, D):
    return np.array([[float(x) for x in r.split(",")] for r in s.split()], np.float64).reshape(-1, D)


def _golden():
    cases = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            blk, L, scale, q, K, V, sel, terms = [c.strip() for c in line.split("|")]
            q = np.array([float(x) for x in q.split(",")])
            D = q.size
            sel = np.zeros(0, np.int32) if sel == "-" else np.array(sel.split(), np.int32)
            xs, vals = [], []
            for t in terms.split():
                x, v = t.split(":")
                xs.append(_term(x))
                vals.append([float(c) for c in v.split(",")])
            cases.append((int(blk), int(L), float(scale), q, _rows(K, D), _rows(V, D), sel,
                          np.array(xs), np.array(vals)))
    return cases


@pytest.mark.parametrize("case", _golden())
def test_tail_worked_by_hand(case):
    blk, L, scale, q, K, V, sel, xs, vals = case
    mK, mV = oracle.block_moments(K, blk), oracle.block_moments(V, blk)
    got = oracle.attend_tail(q, q, K, V, L, blk, scale, sel, mK, mV)
    w = np.exp(xs - xs.max())
    want = (w[:, None] * vals).sum(axis=0) / w.sum()
    np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-15)


def test_block_means_worked_by_hand():
    X = np.array([[0, 1], [1, -1], [1, 0], [0, 0], [-1, 2]], np.float64)
    m = oracle.block_moments(X, 2).astype(np.float64)
    assert m.tolist() == [[0.5, 0.0], [0.5, 0.0], [-1.0, 2.0]]
    X = np.array([[1, 0], [0, 0], [0, 0], [0, 5]], np.float64)
    m = oracle.block_moments(X, 3).astype(np.float64)
    assert m.tolist() == [[R3, 0.0], [0.0, 5.0]]  # the partial block divides by its 1 row


@pytest.mark.parametrize("L", [64, 200, 257])
def test_block_means_match_numpy(L):
    X = RNG.standard_normal((L, 128)) * 3.0
    X[:64] = 1e-4 * RNG.standard_normal((64, 128))  # block 0: means in f16's subnormal range
    got = oracle.block_moments(X, 64)
    nb = (L + 63) // 64
    want = np.stack([X[j * 64:min(L, j * 64 + 64)].mean(axis=0) for j in range(nb)])
    # numpy's mean sums pairwise, the oracle in row order: the f16 roundings agree
    # unless the exact mean sits within a few ulps of binary64 of a rounding boundary
    got16 = got.view(np.uint16).astype(np.int64)
    want16 = want.astype(np.float16).view(np.uint16).astype(np.int64)
    assert np.abs(got16 - want16).max() <= 1
    assert (got16 != want16).mean() < 1e-3


def test_equal_rows_give_the_row():
    row = (RNG.standard_normal(128) * 7).astype(np.float16).astype(np.float64)
    X = np.tile(row, (150, 1))
    m = oracle.block_moments(X, 64)
    assert np.array_equal(m.astype(np.float64), np.tile(row, (3, 1)))


def _cache(dtype, L, Hkv=1, seed=0):
    rng = np.random.default_rng(seed)
    oc = oracle.OracleCache(dtype, 1, Hkv, 128, 64 * ((L + 63) // 64 + 1))
    k = (rng.standard_normal((1, L, Hkv, 128)) * 1.5).astype(np.float16)
    v = rng.standard_normal((1, L, Hkv, 128)).astype(np.float16)
    oc.append(k, v)
    return oc


@pytest.mark.parametrize("dtype", [oracle.F16, oracle.INT8, oracle.Q8_0, oracle.Q4_0])
def test_every_block_listed_is_plain_attention(dtype):
    # nothing is left for the tail: the result is the cache type's own attention,
    # which also pins the binary64 view of the stored rows
    L = 64 * 5 + 17
    oc = _cache(dtype, L, seed=dtype)
    q = (RNG.standard_normal(128) * 2).astype(np.float32)
    sel = np.arange(6, dtype=np.int32)
    got = oc.attend_tail(0, 0, q, 0.09, sel)
    if dtype == oracle.F16:
        want = oracle.attend_f16(q, oc.K[0, 0], oc.V[0, 0], L, 64, 0.09, sel=sel)
    else:
        qc, qs = oracle.quantize_row(q)
        if dtype == oracle.INT8:
            want = oracle.attend_int8(qc, qs, oc.K[0, 0], oc.V[0, 0], oc.ks[0, 0], oc.vs[0, 0],
                                      L, 64, 0.09, sel=sel)
        else:
            att = oracle.attend_q8_0 if dtype == oracle.Q8_0 else oracle.attend_q4_0
            want, _ = att(qc, qs, oc.K[0, 0], oc.V[0, 0], oc.kd[0, 0], oc.vd[0, 0], L, 64, 0.09,
                          sel=sel)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def _equal_key_blocks(L, blk, seed):
    """Rows where every block's keys are one row, and its values come in pairs
    c +- delta around an integer center c (a middle row c when the count is
    odd), so the block means are exact and the tail term is exact too."""
    rng = np.random.default_rng(seed)
    nb = (L + blk - 1) // blk
    K = np.zeros((L, 128))
    V = np.zeros((L, 128))
    for j in range(nb):
        lo, hi = j * blk, min(L, j * blk + blk)
        K[lo:hi] = rng.integers(-4, 5, 128) * 0.25
        c = rng.integers(-3, 4, 128).astype(np.float64)
        m = hi - lo
        for i in range(m // 2):
            delta = rng.integers(0, 4, 128)
            V[lo + 2 * i] = c + delta
            V[lo + 2 * i + 1] = c - delta
        if m % 2:
            V[hi - 1] = c
    return K, V


@pytest.mark.parametrize("sel", [[], [0], [1, 3], [0, 1, 2, 3, 4]])
def test_equal_keys_make_the_tail_exact(sel):
    # all logits of a block are equal, so m e^a at the value mean is exactly the
    # block's own numerator and mass: any listing gives dense attention
    L, blk = 4 * 64 + 37, 64  # the last block (37 rows) is partial
    K, V = _equal_key_blocks(L, blk, 7)
    q = RNG.standard_normal(128).astype(np.float32)
    mK, mV = oracle.block_moments(K, blk), oracle.block_moments(V, blk)
    q64 = q.astype(np.float64)
    got = oracle.attend_tail(q64, q64, K, V, L, blk, 0.3, np.array(sel, np.int32), mK, mV)
    want = oracle.attend_f16(q, K.astype(np.float16), V.astype(np.float16), L, blk, 0.3)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_zero_query_weighs_by_counts():
    # q = 0: a listed token weighs 1 and a left-out block weighs its count, so
    # with exact block means the output is the mean of every value row
    L, blk = 3 * 64 + 9, 64
    _, V = _equal_key_blocks(L, blk, 9)
    K = RNG.standard_normal((L, 128))
    mK, mV = oracle.block_moments(K, blk), oracle.block_moments(V, blk)
    q = np.zeros(128)
    for sel in ([], [2], [0, 3]):
        got = oracle.attend_tail(q, q, K, V, L, blk, 0.7, np.array(sel, np.int32), mK, mV)
        np.testing.assert_allclose(got, V.mean(axis=0), rtol=1e-13, atol=1e-13)
