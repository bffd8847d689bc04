"""Pins of the oracle's sparse-V (eps mode) to facts outside itself (no GPU).

"Sparse Attention -- Quest-style block-selector for long-context decode
(#551)", section "Adaptive tau (the eps mode)": a position's V term is
skipped when its weight is below eps times the running mean weight, and the
page states what that buys: the dropped share of the softmax mass stays
below eps.  Reading R7 takes the mean over the position's 16-token chunk.

Pins: hand-worked keep masks (tests/golden/sparse_v.txt), the mass bound as
an invariant on random heads, eps = 0 against the plain attention functions
(a separate code path), the uniform-logit closed form, and the all-dropped
limit.
"""
import math
import os

import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(5150)
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "sparse_v.txt")


def _logit(s):
    total = 0.0
    for term in s.replace("+", " +").split():
        sign = -1.0 if term.startswith("-") else 1.0
        term = term.lstrip("+-")
        total += sign * (math.log(float(term[2:])) if term.startswith("ln") else float(term))
    return total


def _golden():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            tok, lg, eps, keep = [c.strip() for c in line.split("|")]
            rows.append(([int(x) for x in tok.split()], [_logit(x) for x in lg.split()],
                         float(eps), [bool(int(x)) for x in keep.split()]))
    return rows


@pytest.mark.parametrize("row", _golden())
def test_keep_masks_worked_by_hand(row):
    tok, lg, eps, keep = row
    assert oracle.sparse_v_keep(tok, lg, eps).tolist() == keep


def _f16_head(L, seed, D=128, spread=1.0):
    rng = np.random.default_rng(seed)
    q = (rng.standard_normal(D) * spread).astype(np.float32)
    K = rng.standard_normal((L, D)).astype(np.float16)
    V = rng.standard_normal((L, D)).astype(np.float16)
    return q, K, V


@pytest.mark.parametrize("eps", [0.01, 0.1, 0.5, 1.0, 3.0])
@pytest.mark.parametrize("seed", [1, 2, 3])
def test_dropped_mass_stays_below_eps(eps, seed):
    # the page's guarantee: per chunk every dropped weight is below eps * mean,
    # so the chunk drops less than eps of its mass, and so does the whole head
    L = 700
    q, K, V = _f16_head(L, seed, spread=2.0)
    sel = np.array([0, 3, 4, 7, 10], np.int32)
    full = oracle.attend_f16(q, K, V, L, 64, 128 ** -0.5, sel=sel)
    out, dropped = oracle.attend_f16_sv(q, K, V, L, 64, 128 ** -0.5, eps, sel=sel)
    assert 0.0 <= dropped < eps
    # the numerator lost at most that share of the mass: |out - full| <= dropped * max |v|
    vmax = np.abs(V.astype(np.float64)).max()
    assert np.abs(out - full).max() <= dropped * vmax * (1 + 1e-12) + 1e-15
    if eps >= 1.0:
        assert dropped > 0.0  # something below the mean exists in every chunk here


@pytest.mark.parametrize("dtype", ["f16", "int8"])
def test_eps_zero_is_plain_attention(dtype):
    L = 333
    q, K, V = _f16_head(L, 9)
    sel = np.array([1, 2, 5], np.int32)
    if dtype == "f16":
        want = oracle.attend_f16(q, K, V, L, 64, 0.1, sel=sel)
        got, dropped = oracle.attend_f16_sv(q, K, V, L, 64, 0.1, 0.0, sel=sel)
    else:
        qc, qs = oracle.quantize_row(q)
        Kc = np.zeros((L, 128), np.int8)
        Vc = np.zeros((L, 128), np.int8)
        ks = np.zeros(L, np.float32)
        vs = np.zeros(L, np.float32)
        for t in range(L):
            Kc[t], ks[t] = oracle.quantize_row(K[t].astype(np.float32))
            Vc[t], vs[t] = oracle.quantize_row(V[t].astype(np.float32))
        want = oracle.attend_int8(qc, qs, Kc, Vc, ks, vs, L, 64, 0.1, sel=sel)
        got, dropped = oracle.attend_int8_sv(qc, qs, Kc, Vc, ks, vs, L, 64, 0.1, 0.0, sel=sel)
    assert dropped == 0.0
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-15)


def test_uniform_logits_closed_form():
    # q = 0: every weight is 1 and equals its chunk mean, so eps <= 1 drops
    # nothing (the output is the mean of the attended values) and any eps > 1
    # drops everything (the output is zero, the mass share dropped is 1)
    L = 200
    _, K, V = _f16_head(L, 4)
    q = np.zeros(128, np.float32)
    mean_v = V[:L].astype(np.float64).mean(axis=0)
    out, dropped = oracle.attend_f16_sv(q, K, V, L, 64, 0.3, 1.0)
    assert dropped == 0.0
    np.testing.assert_allclose(out, mean_v, rtol=0, atol=1e-14)
    out, dropped = oracle.attend_f16_sv(q, K, V, L, 64, 0.3, 1.0 + 1e-9)
    assert dropped == 1.0 and not out.any()


def test_eps_above_chunk_size_drops_everything():
    # p_t <= sum over its chunk = |c| * mean < eps * mean once eps > |c| (16)
    L = 256
    q, K, V = _f16_head(L, 6, spread=3.0)
    out, dropped = oracle.attend_f16_sv(q, K, V, L, 64, 128 ** -0.5, 16.5)
    assert dropped == 1.0 and not out.any()
