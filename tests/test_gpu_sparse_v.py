"""GPU sparse-V (eps mode) decode vs the oracle.

Bar: relative L2 per (sequence, query head) within 2e-3 (f16) / 8e-3 (int8)
and within 1e-4 against the oracle's attention with the same rule, on the
GPU's own block selection; eps = 0 bit-identical to the plain decode.

The keep decision compares a weight with eps times its chunk mean; the GPU
takes it in f32, the oracle in fp64.  A position within rounding of its
threshold may fall on either side, and both outcomes are correct.  The test
finds those positions (relative margin below 1e-4, from the oracle's fp64
logits) and widens the bar by the most they can move the output:
sum over them of w_t |v_t| / Z, relative to |out|.
"""
import numpy as np
import pytest
import torch

import long_context_decode_kv_gb300 as kvd
import oracle
from gpu_util import TIGHT, TOL, assert_outputs, dev, make_pair, rel_l2_rows, scale_for, seeded

pytestmark = pytest.mark.gpu
CHUNK = 16


def _tokens(L, sel):
    if sel is None:
        return np.arange(L)
    return np.concatenate([np.arange(b * 64, min(b * 64 + 64, L)) for b in sel]) if len(sel) \
        else np.zeros(0, np.int64)


def _codes(dtype, rows):
    """Integer code values of cache rows: int8 codes, or 4-bit codes minus 8."""
    if dtype == kvd.Q4_0:
        out = np.empty(rows.shape[:-1] + (rows.shape[-1] * 2,), np.float64)
        out[..., 0::2] = (rows & 15).astype(np.float64) - 8
        out[..., 1::2] = (rows >> 4).astype(np.float64) - 8
        return out
    return rows.astype(np.float64)


def _logits(dtype, oc, qh, b, g, tok, scale):
    if dtype == kvd.F16:
        K = oc.K[b, g, tok].astype(np.float64)
        return scale * (K @ qh.astype(np.float64))
    qc, qs = oracle.quantize_row(qh)
    if dtype in (kvd.Q8_0, kvd.Q4_0):
        K = _codes(dtype, oc.K[b, g, tok]) * np.repeat(
            oc.kd[b, g, tok].astype(np.float64), 32, axis=1)
        return (K @ qc.astype(np.float64)) * float(qs) * scale
    dots = oracle.qk_int8(qc, oc.K[b, g, tok])
    return dots.astype(np.float64) * float(qs) * oc.ks[b, g, tok].astype(np.float64) * scale


def _ambiguity(tok, lg, vrows, eps):
    """Output shift (L2) that positions at their threshold may cause."""
    if eps == 0 or len(tok) == 0:
        return 0.0
    w = np.exp(lg - lg.max())
    amb = np.zeros(len(tok), bool)
    for c in np.unique(tok // CHUNK):
        m = tok // CHUNK == c
        p = np.exp(lg[m] - lg[m].max())
        thr = eps * p.sum() / m.sum()
        amb[m] = np.abs(p / thr - 1.0) < 1e-4
    return float((w[amb] * np.linalg.norm(vrows[amb], axis=1)).sum() / w.sum())


def _reference(dtype, oc, q_np, b, g, G, L, sel, eps, scale):
    outs, drops, slack = [], [], []
    tok = _tokens(L, sel)
    if dtype == kvd.F16:
        vrows = oc.V[b, g, tok].astype(np.float64)
    elif dtype in (kvd.Q8_0, kvd.Q4_0):
        vrows = _codes(dtype, oc.V[b, g, tok]) * np.repeat(
            oc.vd[b, g, tok].astype(np.float64), 32, axis=1)
    else:
        vrows = oc.V[b, g, tok].astype(np.float64) * oc.vs[b, g, tok, None].astype(np.float64)
    for h in range(G):
        qh = q_np[b, g * G + h]
        if dtype == kvd.F16:
            o, d = oracle.attend_f16_sv(qh, oc.K[b, g], oc.V[b, g], L, 64, scale, eps, sel=sel)
        elif dtype in (kvd.Q8_0, kvd.Q4_0):
            qc, qs = oracle.quantize_row(qh)
            att = oracle.attend_q8_0 if dtype == kvd.Q8_0 else oracle.attend_q4_0
            o, d = att(qc, qs, oc.K[b, g], oc.V[b, g], oc.kd[b, g], oc.vd[b, g], L, 64, scale,
                       sel=sel, eps=eps)
        else:
            qc, qs = oracle.quantize_row(qh)
            o, d = oracle.attend_int8_sv(qc, qs, oc.K[b, g], oc.V[b, g], oc.ks[b, g],
                                         oc.vs[b, g], L, 64, scale, eps, sel=sel)
        shift = _ambiguity(tok, _logits(dtype, oc, qh, b, g, tok, scale), vrows, eps)
        outs.append(o)
        drops.append(d)
        slack.append(shift / max(np.linalg.norm(o), 1e-300))
    return np.stack(outs), drops, np.array(slack)


def _assert_close(gpu, ref, slack, dtype, what):
    e = rel_l2_rows(gpu, ref)
    assert np.all(np.isfinite(e)), what
    bar = np.minimum(TOL[dtype], TIGHT) + slack
    assert np.all(e <= bar), f"{what}: rel L2 {e.max():.3e} over {bar[np.argmax(e - bar)]:.3e}"


def _case(dtype, B, Hkv, G, L, seed):
    k = seeded((B, L, Hkv, 128), seed, scale=1.5)
    v = seeded((B, L, Hkv, 128), seed + 1)
    gc, oc = make_pair(dtype, k, v)
    q = seeded((B, Hkv * G, 128), seed + 2, scale=2.0, dtype=torch.float32)
    return gc, oc, q


@pytest.mark.parametrize("dtype", [kvd.F16, kvd.INT8, kvd.Q8_0, kvd.Q4_0])
@pytest.mark.parametrize("eps", [0.05, 0.5, 2.0])
@pytest.mark.parametrize("sparse", [True, False])
def test_sparse_v_matches_oracle(dtype, eps, sparse):
    B, Hkv, G, L = 2, 2, 4, 64 * 37 + 21  # ragged: the last block and chunk are partial
    gc, oc, q = _case(dtype, B, Hkv, G, L, 300 + int(10 * eps) + int(sparse))
    ws = kvd.make_workspace(gc, Hkv * G)
    sel_idx = sel_cnt = None
    max_sel = 0
    if sparse:
        nbmax = gc.max_seq // 64
        sel_idx = torch.zeros((B, Hkv, nbmax), dtype=torch.int32, device=dev())
        sel_cnt = torch.zeros((B, Hkv), dtype=torch.int32, device=dev())
        kvd.select_blocks(gc, q, 9, 4, 100, sel_idx, sel_cnt, ws)
        max_sel = kvd.selected_count(L, 9, 4, 100)
    out = torch.full((B, Hkv * G, 128), float("nan"), device=dev())
    kvd.decode_attn_sv(gc, q, scale_for(), sel_idx, sel_cnt, max_sel, eps, out, ws)
    torch.cuda.synchronize()
    q_np = q.cpu().numpy()
    dropped = []
    for b in range(B):
        for g in range(Hkv):
            sel = None
            if sparse:
                sel = sel_idx[b, g, :int(sel_cnt[b, g])].cpu().numpy()
            ref, d, slack = _reference(dtype, oc, q_np, b, g, G, L, sel, eps, scale_for())
            dropped += d
            _assert_close(out[b, g * G:(g + 1) * G], ref, slack, dtype,
                          f"sv {dtype} eps {eps} sparse {sparse} b{b} g{g}")
    assert max(dropped) < eps
    if eps >= 0.5:
        assert min(dropped) > 0.0  # the rule did drop something in every head


@pytest.mark.parametrize("dtype", [kvd.F16, kvd.INT8, kvd.Q8_0, kvd.Q4_0])
def test_eps_zero_is_bit_identical(dtype):
    B, Hkv, G, L = 1, 8, 4, 9000
    gc, oc, q = _case(dtype, B, Hkv, G, L, 350)
    ws = kvd.make_workspace(gc, Hkv * G)
    nbmax = gc.max_seq // 64
    sel_idx = torch.zeros((B, Hkv, nbmax), dtype=torch.int32, device=dev())
    sel_cnt = torch.zeros((B, Hkv), dtype=torch.int32, device=dev())
    kvd.select_blocks(gc, q, 30, 4, 256, sel_idx, sel_cnt, ws)
    max_sel = kvd.selected_count(L, 30, 4, 256)
    a = torch.empty((B, Hkv * G, 128), device=dev())
    b_ = torch.empty_like(a)
    kvd.decode_attn(gc, q, scale_for(), sel_idx, sel_cnt, max_sel, a, ws)
    kvd.decode_attn_sv(gc, q, scale_for(), sel_idx, sel_cnt, max_sel, 0.0, b_, ws)
    c = torch.empty_like(a)
    d = torch.empty_like(a)
    kvd.decode_attn_dense(gc, q, scale_for(), c, ws)
    kvd.decode_attn_sv(gc, q, scale_for(), None, None, 0, 0.0, d, ws)
    torch.cuda.synchronize()
    assert torch.equal(a, b_) and torch.equal(c, d)


@pytest.mark.parametrize("dtype", [kvd.F16, kvd.INT8])
def test_uniform_logits_and_drop_all(dtype):
    # q = 0: every weight equals its chunk mean, so eps <= 1 keeps every V term
    # (the output is the mean of the values) and eps > 1 drops all of them
    B, Hkv, G, L = 1, 2, 2, 1000
    gc, oc, _ = _case(dtype, B, Hkv, G, L, 360)
    q = torch.zeros((B, Hkv * G, 128), dtype=torch.float32, device=dev())
    ws = kvd.make_workspace(gc, Hkv * G)
    out = torch.full((B, Hkv * G, 128), float("nan"), device=dev())
    kvd.decode_attn_sv(gc, q, scale_for(), None, None, 0, 1.0, out, ws)
    torch.cuda.synchronize()
    for g in range(Hkv):
        if dtype == kvd.F16:
            mean_v = oc.V[0, g, :L].astype(np.float64).mean(axis=0)
        else:
            mean_v = (oc.V[0, g, :L].astype(np.float64) *
                      oc.vs[0, g, :L, None].astype(np.float64)).mean(axis=0)
        assert_outputs(out[0, g * G:(g + 1) * G], np.stack([mean_v] * G), dtype, "uniform")
    kvd.decode_attn_sv(gc, q, scale_for(), None, None, 0, 1.5, out, ws)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0


def test_invalid_eps_rejected_on_host():
    gc = kvd.KVCache(kvd.F16, 1, 1, 128, device=dev())
    k = seeded((1, 10, 1, 128), 1)
    kvd.kv_append(gc, k, k)
    q = torch.zeros((1, 1, 128), device=dev())
    out = torch.zeros_like(q)
    ws = kvd.make_workspace(gc, 1)
    for bad in (-0.1, float("nan"), float("inf")):
        with pytest.raises(kvd.KvdError):
            kvd.decode_attn_sv(gc, q, 0.1, None, None, 0, bad, out, ws)
