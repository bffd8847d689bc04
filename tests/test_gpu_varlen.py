"""Per-sequence lengths in one batch vs the oracle, one oracle cache per
sequence (each sequence is an independent problem of its own length).

Bars as for a single length: rows, codes, scales and bounds bit-exact after a
per-sequence append; each (sequence, KV head) list identical to the oracle's on
that sequence's own length up to the tie window; outputs within the cache
type's bar and 1e-4 of the oracle on the GPU's lists; a sequence of length 0
selects nothing and outputs zeros.
"""
import numpy as np
import pytest
import torch

import long_context_decode_kv_gb300 as kvd
import oracle
from gpu_util import TIE_REL, assert_outputs, dev, scale_for, seeded
from test_gpu_append import _compare

pytestmark = pytest.mark.gpu
LENS = [70, 1000, 0, 2389, 1, 640]


def _build(dtype, lens, Hkv, G, seed, moments=False):
    B = len(lens)
    max_seq = (max(lens) + 200 + 63) // 64 * 64
    gc = kvd.KVCache(dtype, B, Hkv, max_seq, device=dev(), moments=moments)
    ocs = []
    for b, L in enumerate(lens):
        oc = oracle.OracleCache(dtype, 1, Hkv, 128, max_seq, 64)
        if L:
            k = seeded((1, L, Hkv, 128), seed + 7 * b, scale=1.5)
            v = seeded((1, L, Hkv, 128), seed + 7 * b + 1)
            kvd.kv_append(gc.view(b), k, v)
            oc.append(k.cpu().numpy(), v.cpu().numpy())
        ocs.append(oc)
    lens_t = torch.tensor(lens, dtype=torch.int32, device=dev())
    gc.set_seq_lens(lens_t)
    gc.len = max(lens)
    q = seeded((B, Hkv * G, 128), seed + 99, scale=2.0, dtype=torch.float32)
    torch.cuda.synchronize()
    return gc, ocs, q, lens_t


def _oracle_head(dtype, oc, qh, g, sel):
    L = oc.len
    if L == 0:
        return np.zeros(128)
    if dtype == kvd.F16:
        return oracle.attend_f16(qh, oc.K[0, g], oc.V[0, g], L, 64, scale_for(), sel=sel)
    qc, qs = oracle.quantize_row(qh)
    if dtype == kvd.INT8:
        return oracle.attend_int8(qc, qs, oc.K[0, g], oc.V[0, g], oc.ks[0, g], oc.vs[0, g], L,
                                  64, scale_for(), sel=sel)
    att = oracle.attend_q8_0 if dtype == kvd.Q8_0 else oracle.attend_q4_0
    return att(qc, qs, oc.K[0, g], oc.V[0, g], oc.kd[0, g], oc.vd[0, g], L, 64, scale_for(),
               sel=sel)[0]


def _check_lists(idx, cnt, ocs, q_np, k_sel, sink, recent, G, per_head=False):
    for b, oc in enumerate(ocs):
        L = oc.len
        nb = (L + 63) // 64
        rows = range(cnt.shape[1])
        for r in rows:
            g = r // G if per_head else r
            qh = q_np[b, r][None] if per_head else q_np[b, g * G:(g + 1) * G]
            n = int(cnt[b, r])
            if L == 0:
                assert n == 0
                continue
            ub, _, mag = oracle.block_scores(qh, oc.kmin[0, g, :nb], oc.kmax[0, g, :nb])
            want, kth = oracle.select(L, 64, ub, k_sel, sink, recent)
            got = idx[b, r, :n]
            assert n == len(want), (b, r, n, len(want))
            assert np.all(np.diff(got) > 0)
            se, rb = oracle.forced_range(L, 64, sink, recent)
            for j in set(got.tolist()) ^ set(want.tolist()):
                assert se <= j < rb
                assert abs(ub[j] - kth) <= TIE_REL * max(abs(kth), mag[j]), (b, r, j)


@pytest.mark.parametrize("dtype", [kvd.F16, kvd.INT8, kvd.Q4_0])
@pytest.mark.parametrize("G", [1, 4])
@pytest.mark.parametrize("k_sel,sink,recent", [(5, 4, 100), (0, 64, 64), (10 ** 6, 4, 64),
                                               (3, 0, 0)])
def test_varlen_select_and_decode(dtype, G, k_sel, sink, recent):
    Hkv = 2
    gc, ocs, q, _ = _build(dtype, LENS, Hkv, G, 700 + G)
    B = len(LENS)
    ws = kvd.make_workspace(gc, Hkv * G)
    nbmax = gc.max_seq // 64
    sel_idx = torch.full((B, Hkv, nbmax), -5, dtype=torch.int32, device=dev())
    sel_cnt = torch.full((B, Hkv), -5, dtype=torch.int32, device=dev())
    kvd.select_blocks(gc, q, k_sel, sink, recent, sel_idx, sel_cnt, ws)
    max_sel = kvd.selected_count(max(LENS), k_sel, sink, recent)
    out = torch.full((B, Hkv * G, 128), float("nan"), device=dev())
    dense = torch.full_like(out, float("nan"))
    kvd.decode_attn(gc, q, scale_for(), sel_idx, sel_cnt, max_sel, out, ws)
    kvd.decode_attn_dense(gc, q, scale_for(), dense, ws)
    torch.cuda.synchronize()
    assert gc.device_status() == 0
    q_np = q.cpu().numpy()
    idx, cnt = sel_idx.cpu().numpy(), sel_cnt.cpu().numpy()
    _check_lists(idx, cnt, ocs, q_np, k_sel, sink, recent, G)
    for b, oc in enumerate(ocs):
        for g in range(Hkv):
            sel = idx[b, g, :cnt[b, g]]
            ref = np.stack([_oracle_head(dtype, oc, q_np[b, g * G + h], g, sel)
                            for h in range(G)])
            dref = np.stack([_oracle_head(dtype, oc, q_np[b, g * G + h], g, None)
                             for h in range(G)])
            if oc.len == 0:
                assert not out[b, g * G:(g + 1) * G].any()
                assert not dense[b, g * G:(g + 1) * G].any()
                continue
            assert_outputs(out[b, g * G:(g + 1) * G], ref, dtype, f"varlen b{b} g{g}")
            assert_outputs(dense[b, g * G:(g + 1) * G], dref, dtype, f"varlen dense b{b} g{g}")


@pytest.mark.parametrize("dtype", [kvd.F16, kvd.INT8, kvd.Q8_0, kvd.Q4_0])
@pytest.mark.parametrize("n_new", [1, 5, 70])
def test_varlen_append(dtype, n_new):
    # each sequence's new rows land at its own position, and the bounds of
    # its partial last block merge with its own earlier rows
    Hkv = 3
    gc, ocs, _, lens_t = _build(dtype, LENS, Hkv, 1, 750, moments=True)
    k = seeded((len(LENS), n_new, Hkv, 128), 760, scale=2.0)
    v = seeded((len(LENS), n_new, Hkv, 128), 761)
    kvd.kv_append(gc, k, v)
    lens_t += n_new
    torch.cuda.synchronize()
    assert gc.len == max(LENS) + n_new and gc.device_status() == 0
    kh, vh = k.cpu().numpy(), v.cpu().numpy()
    for b, oc in enumerate(ocs):
        oc.append(kh[b:b + 1], vh[b:b + 1])
        _compare(gc.view(b), oc)
        nb = (oc.len + 63) // 64
        got = gc.moments[b, :, :nb].cpu().numpy()
        for h in range(Hkv):
            mK, mV = oc.moments(0, h)
            for i, want in enumerate((mK, mV)):
                step = np.spacing(np.abs(want)).astype(np.float64)
                assert np.all(np.abs(got[h, :, i].astype(np.float64) - want) <= step)


def test_varlen_per_head_and_tail():
    dtype, Hkv, G = kvd.INT8, 2, 4
    gc, ocs, q, _ = _build(dtype, LENS, Hkv, G, 780, moments=True)
    B = len(LENS)
    ws = kvd.make_workspace(gc, Hkv * G)
    nbmax = gc.max_seq // 64
    # per-head lists on each sequence's own length
    h_idx = torch.full((B, Hkv * G, nbmax), -5, dtype=torch.int32, device=dev())
    h_cnt = torch.full((B, Hkv * G), -5, dtype=torch.int32, device=dev())
    kvd.select_blocks_per_head(gc, q, 4, 4, 64, h_idx, h_cnt, ws)
    # the moment tail of the shared lists
    s_idx = torch.zeros((B, Hkv, nbmax), dtype=torch.int32, device=dev())
    s_cnt = torch.zeros((B, Hkv), dtype=torch.int32, device=dev())
    kvd.select_blocks(gc, q, 4, 4, 64, s_idx, s_cnt, ws)
    max_sel = kvd.selected_count(max(LENS), 4, 4, 64)
    tail = torch.full((B, Hkv * G, 128), float("nan"), device=dev())
    kvd.decode_attn_tail(gc, q, scale_for(), s_idx, s_cnt, max_sel, tail, ws)
    torch.cuda.synchronize()
    assert gc.device_status() == 0
    q_np = q.cpu().numpy()
    _check_lists(h_idx.cpu().numpy(), h_cnt.cpu().numpy(), ocs, q_np, 4, 4, 64, G,
                 per_head=True)
    idx, cnt = s_idx.cpu().numpy(), s_cnt.cpu().numpy()
    for b, oc in enumerate(ocs):
        for g in range(Hkv):
            if oc.len == 0:
                assert not tail[b, g * G:(g + 1) * G].any()
                continue
            sel = idx[b, g, :cnt[b, g]]
            ref = np.stack([oc.attend_tail(0, g, q_np[b, g * G + h], scale_for(), sel)
                            for h in range(G)])
            assert_outputs(tail[b, g * G:(g + 1) * G], ref, dtype, f"varlen tail b{b} g{g}")


def test_lengths_past_len_are_reported():
    gc, ocs, q, lens_t = _build(kvd.F16, [100, 200], 1, 1, 790)
    lens_t[1] = 10 ** 6  # past len: clamped to len and reported
    ws = kvd.make_workspace(gc, 1)
    out = torch.empty((2, 1, 128), device=dev())
    kvd.decode_attn_dense(gc, q, scale_for(), out, ws)
    torch.cuda.synchronize()
    assert kvd.STATUS[gc.device_status()] == "KVD_ERR_INVALID"


@pytest.mark.parametrize("dtype", [kvd.F16, kvd.INT8])
@pytest.mark.parametrize("k_sel", [4, -1])
def test_varlen_decode_steps(dtype, k_sel):
    # kvd_decode_step appends each sequence's token at its own length and
    # attends that length + 1; the caller then advances the lengths
    Hkv, G = 2, 4
    lens = [70, 1000, 0, 2389, 63]
    gc, ocs, _, lens_t = _build(dtype, lens, Hkv, G, 800)
    B = len(lens)
    ws = kvd.make_workspace(gc, Hkv * G)
    nbmax = gc.max_seq // 64
    sel_idx = torch.zeros((B, Hkv, nbmax), dtype=torch.int32, device=dev())
    sel_cnt = torch.zeros((B, Hkv), dtype=torch.int32, device=dev())
    out = torch.empty((B, Hkv * G, 128), device=dev())
    for step in range(3):
        q = seeded((B, Hkv * G, 128), 810 + step, scale=2.0, dtype=torch.float32)
        kn = seeded((B, 1, Hkv, 128), 820 + step)
        vn = seeded((B, 1, Hkv, 128), 830 + step)
        kvd.decode_step(gc, q, kn, vn, scale_for(), k_sel, 4, 64, out, ws, sel_idx, sel_cnt)
        lens_t += 1
        torch.cuda.synchronize()
        assert gc.device_status() == 0
        q_np = q.cpu().numpy()
        idx, cnt = sel_idx.cpu().numpy(), sel_cnt.cpu().numpy()
        for b, oc in enumerate(ocs):
            oc.append(kn[b:b + 1].cpu().numpy(), vn[b:b + 1].cpu().numpy())
            for g in range(Hkv):
                sel = None if k_sel < 0 else idx[b, g, :cnt[b, g]]
                ref = np.stack([_oracle_head(dtype, oc, q_np[b, g * G + h], g, sel)
                                for h in range(G)])
                assert_outputs(out[b, g * G:(g + 1) * G], ref, dtype, f"step{step} b{b} g{g}")
        if k_sel >= 0:
            _check_lists(idx, cnt, ocs, q_np, k_sel, 4, 64, G)
    assert gc.len == max(lens) + 3
