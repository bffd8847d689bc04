"""GPU moment tail vs the oracle.

"SCSA: Self-Calibrating Subquadratic Attention", "2. Mechanism": every block
the selection leaves out still contributes m exp(scale q . c_K) at its value
mean c_V inside the shared normalizer (the oracle's reading R10).

Bars:
  * block means: within one binary16 step of the oracle's (the GPU sums the
    f32 rows in token order, the oracle in binary64, and both round once);
  * outputs: relative L2 per (sequence, query head) within the cache type's
    bar and within 1e-4 of the oracle's tail attention on the GPU's own
    selection;
  * every block listed: bit-identical to the plain decode.
"""
import numpy as np
import pytest
import torch

import long_context_decode_kv_gb300 as kvd
import oracle
from long_context_decode_kv_gb300 import synth
from gpu_util import TOL, assert_outputs, dev, make_pair, scale_for, seeded

pytestmark = pytest.mark.gpu
DTYPES = [kvd.F16, kvd.INT8, kvd.Q8_0, kvd.Q4_0]


def _moments_close(gc, oc, what):
    nb = (oc.len + 63) // 64
    got = gc.moments[..., :nb, :, :].cpu().numpy()  # [B, Hkv, nb, 2, 128]
    for b in range(oc.B):
        for h in range(oc.Hkv):
            mK, mV = oc.moments(b, h)
            for i, want in enumerate((mK, mV)):
                g = got[b, h, :, i].astype(np.float64)
                w = want.astype(np.float64)
                step = np.spacing(np.abs(want)).astype(np.float64)  # one f16 step
                bad = np.abs(g - w) > step * (1 + 1e-9)
                assert not bad.any(), (what, b, h, i, np.argwhere(bad)[:4])
                # and nearly always equal
                assert (g != w).mean() < 0.01, (what, b, h, i, (g != w).mean())


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("chunks", [[200], [1] * 70 + [130], [63, 1, 64, 72]])
def test_block_means_after_append(dtype, chunks):
    B, Hkv, L = 2, 3, sum(chunks)
    k = seeded((B, L, Hkv, 128), 11, scale=1.5)
    v = seeded((B, L, Hkv, 128), 12)
    gc, oc = make_pair(dtype, k, v, chunks=chunks, moments=True)
    _moments_close(gc, oc, f"{dtype} {chunks[:3]}")


@pytest.mark.parametrize("dtype", DTYPES)
def test_block_means_after_rewind(dtype):
    # rewinding len into a block and appending other rows recomputes its means
    B, Hkv = 1, 2
    k = seeded((B, 150, Hkv, 128), 21)
    v = seeded((B, 150, Hkv, 128), 22)
    gc, oc = make_pair(dtype, k, v, moments=True)
    gc.len = 100
    k2 = seeded((B, 40, Hkv, 128), 23, scale=3.0)
    v2 = seeded((B, 40, Hkv, 128), 24, scale=3.0)
    kvd.kv_append(gc, k2, v2)
    torch.cuda.synchronize()
    oc2 = oracle.OracleCache(dtype, B, Hkv, 128, oc.max_seq, 64)
    oc2.append(k[:, :100].cpu().numpy(), v[:, :100].cpu().numpy())
    oc2.append(k2.cpu().numpy(), v2.cpu().numpy())
    _moments_close(gc, oc2, f"rewind {dtype}")


def _case(dtype, B, Hkv, G, L, seed):
    k = seeded((B, L, Hkv, 128), seed, scale=1.5)
    v = seeded((B, L, Hkv, 128), seed + 1)
    gc, oc = make_pair(dtype, k, v, moments=True)
    q = seeded((B, Hkv * G, 128), seed + 2, scale=2.0, dtype=torch.float32)
    return gc, oc, q


def _check(gc, oc, q, sel_idx, sel_cnt, out, G, dtype, what):
    q_np = q.cpu().numpy()
    idx = sel_idx.cpu().numpy()
    cnt = sel_cnt.cpu().numpy()
    for b in range(oc.B):
        for g in range(oc.Hkv):
            sel = idx[b, g, :cnt[b, g]]
            ref = np.stack([oc.attend_tail(b, g, q_np[b, g * G + h], scale_for(), sel)
                            for h in range(G)])
            assert_outputs(out[b, g * G:(g + 1) * G], ref, dtype, f"{what} b{b} g{g}")


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_tail_matches_oracle(dtype, G):
    B, Hkv, L = 2, 2, 64 * 37 + 21  # ragged: the last block is partial
    gc, oc, q = _case(dtype, B, Hkv, G, L, 400 + G)
    ws = kvd.make_workspace(gc, Hkv * G)
    nbmax = gc.max_seq // 64
    sel_idx = torch.zeros((B, Hkv, nbmax), dtype=torch.int32, device=dev())
    sel_cnt = torch.zeros((B, Hkv), dtype=torch.int32, device=dev())
    # recent 0: the partial last block can fall to the tail too
    kvd.select_blocks(gc, q, 6, 4, 0, sel_idx, sel_cnt, ws)
    max_sel = kvd.selected_count(L, 6, 4, 0)
    out = torch.full((B, Hkv * G, 128), float("nan"), device=dev())
    kvd.decode_attn_tail(gc, q, scale_for(), sel_idx, sel_cnt, max_sel, out, ws)
    torch.cuda.synchronize()
    _check(gc, oc, q, sel_idx, sel_cnt, out, G, dtype, f"tail {dtype} G{G}")
    assert gc.device_status() == 0


@pytest.mark.parametrize("dtype", DTYPES)
def test_tail_over_hand_made_lists(dtype):
    # empty rows (everything in the tail), single blocks, the last block alone,
    # and a long list spanning many 32-entry loads of the producer's walk
    B, Hkv, G, L = 1, 6, 4, 64 * 300 + 5
    gc, oc, q = _case(dtype, B, Hkv, G, L, 450)
    ws = kvd.make_workspace(gc, Hkv * G)
    nb = (L + 63) // 64
    nbmax = gc.max_seq // 64
    rows = [[], [0], [nb - 1], list(range(0, nb, 3)), list(range(40, 160)),
            sorted(np.random.default_rng(5).choice(nb, 200, replace=False).tolist())]
    sel_idx = torch.zeros((B, Hkv, nbmax), dtype=torch.int32)
    sel_cnt = torch.zeros((B, Hkv), dtype=torch.int32)
    for g, r in enumerate(rows):
        sel_idx[0, g, :len(r)] = torch.tensor(r, dtype=torch.int32)
        sel_cnt[0, g] = len(r)
    sel_idx, sel_cnt = sel_idx.to(dev()), sel_cnt.to(dev())
    out = torch.full((B, Hkv * G, 128), float("nan"), device=dev())
    kvd.decode_attn_tail(gc, q, scale_for(), sel_idx, sel_cnt, max(len(r) for r in rows), out,
                         ws)
    torch.cuda.synchronize()
    _check(gc, oc, q, sel_idx, sel_cnt, out, G, dtype, f"lists {dtype}")


@pytest.mark.parametrize("dtype", DTYPES)
def test_every_block_listed_is_plain_decode(dtype):
    B, Hkv, G, L = 1, 8, 4, 9000
    gc, oc, q = _case(dtype, B, Hkv, G, L, 470)
    ws = kvd.make_workspace(gc, Hkv * G)
    nb = (L + 63) // 64
    nbmax = gc.max_seq // 64
    sel_idx = torch.zeros((B, Hkv, nbmax), dtype=torch.int32, device=dev())
    sel_idx[..., :nb] = torch.arange(nb, dtype=torch.int32, device=dev())
    sel_cnt = torch.full((B, Hkv), nb, dtype=torch.int32, device=dev())
    a = torch.empty((B, Hkv * G, 128), device=dev())
    b_ = torch.empty_like(a)
    kvd.decode_attn(gc, q, scale_for(), sel_idx, sel_cnt, nb, a, ws)
    kvd.decode_attn_tail(gc, q, scale_for(), sel_idx, sel_cnt, nb, b_, ws)
    torch.cuda.synchronize()
    assert torch.equal(a, b_)


@pytest.mark.parametrize("k_sel", [16, 126])
def test_tail_moves_toward_dense(k_sel):
    # on the 32K GQA recipe the tail gives back part of what the selection
    # leaves out: its error against dense attention is smaller
    w = synth.QWEN3_32K
    q, k, v, _ = synth.make_workload(w, device=dev())
    gc = kvd.KVCache(w.dtype, w.B, w.Hkv, w.L + 64, device=dev(), moments=True)
    kvd.kv_append(gc, k, v)
    ws = kvd.make_workspace(gc, q.shape[1])
    B, Hkv = gc.batch, gc.n_kv_heads
    nbmax = gc.max_seq // 64
    sel_idx = torch.zeros((B, Hkv, nbmax), dtype=torch.int32, device=dev())
    sel_cnt = torch.zeros((B, Hkv), dtype=torch.int32, device=dev())
    kvd.select_blocks(gc, q, k_sel, w.sink_tokens, w.recent_tokens, sel_idx, sel_cnt, ws)
    max_sel = kvd.selected_count(gc.len, k_sel, w.sink_tokens, w.recent_tokens)
    dense, sparse, tail = (torch.empty_like(q) for _ in range(3))
    kvd.decode_attn_dense(gc, q, scale_for(), dense, ws)
    kvd.decode_attn(gc, q, scale_for(), sel_idx, sel_cnt, max_sel, sparse, ws)
    kvd.decode_attn_tail(gc, q, scale_for(), sel_idx, sel_cnt, max_sel, tail, ws)
    torch.cuda.synchronize()
    e_sparse = ((sparse - dense).norm(dim=-1) / dense.norm(dim=-1)).median().item()
    e_tail = ((tail - dense).norm(dim=-1) / dense.norm(dim=-1)).median().item()
    assert e_tail < e_sparse, (e_tail, e_sparse)


@pytest.mark.parametrize("dtype", [kvd.F16, kvd.INT8])
@pytest.mark.parametrize("k_sel", [3, -1])
def test_decode_steps_keep_block_means(dtype, k_sel):
    # a decode step appends through the append kernel when the cache keeps
    # block means (sparse and dense arms), so the means stay current
    B, Hkv, G, L = 1, 2, 4, 64 * 6 + 60
    k = seeded((B, L, Hkv, 128), 31)
    v = seeded((B, L, Hkv, 128), 32)
    gc, oc = make_pair(dtype, k, v, moments=True)
    ws = kvd.make_workspace(gc, Hkv * G)
    out = torch.empty((B, Hkv * G, 128), device=dev())
    for step in range(6):  # crosses into a new block
        q = seeded((B, Hkv * G, 128), 40 + step, dtype=torch.float32)
        kn = seeded((B, 1, Hkv, 128), 50 + step)
        vn = seeded((B, 1, Hkv, 128), 60 + step)
        kvd.decode_step(gc, q, kn, vn, scale_for(), k_sel, 4, 64, out, ws)
        oc.append(kn.cpu().numpy(), vn.cpu().numpy())
    torch.cuda.synchronize()
    assert gc.len == oc.len
    _moments_close(gc, oc, f"steps {dtype} {k_sel}")
