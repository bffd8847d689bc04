"""GPU per-query-head selection and decode vs the oracle (the ablation of the
GQA-shared selection: "Certified Sparse Attention via Perturbed Retrieval",
Appendix Table 4, one scan per query head).

Bars as for the shared path: each head's list identical to the oracle's top-K
on that head's own bound except blocks within 1e-5 (relative) of its K-th
bound; outputs within the cache type's bar and 1e-4 of the oracle on the
GPU's lists.  With one query head per KV head both paths are the same
computation, bit for bit.
"""
import numpy as np
import pytest
import torch

import long_context_decode_kv_gb300 as kvd
import oracle
from gpu_util import TIE_REL, assert_outputs, dev, make_pair, scale_for, seeded

pytestmark = pytest.mark.gpu


def _case(dtype, B, Hkv, G, L, seed):
    k = seeded((B, L, Hkv, 128), seed, scale=1.5)
    v = seeded((B, L, Hkv, 128), seed + 1)
    gc, oc = make_pair(dtype, k, v)
    q = seeded((B, Hkv * G, 128), seed + 2, scale=2.0, dtype=torch.float32)
    return gc, oc, q


def _select(gc, q, k_sel, sink, recent, ws):
    B, H = q.shape[0], q.shape[1]
    nbmax = gc.max_seq // 64
    sel_idx = torch.full((B, H, nbmax), -7, dtype=torch.int32, device=dev())
    sel_cnt = torch.full((B, H), -7, dtype=torch.int32, device=dev())
    kvd.select_blocks_per_head(gc, q, k_sel, sink, recent, sel_idx, sel_cnt, ws)
    return sel_idx, sel_cnt


def _check_lists(sel_idx, sel_cnt, oc, q_np, k_sel, sink, recent, G):
    L = oc.len
    nb = (L + 63) // 64
    idx, cnt = sel_idx.cpu().numpy(), sel_cnt.cpu().numpy()
    B, H = cnt.shape
    for b in range(B):
        for h in range(H):
            g = h // G
            ub, _, mag = oracle.block_scores(q_np[b, h][None], oc.kmin[b, g, :nb],
                                             oc.kmax[b, g, :nb])
            want, kth = oracle.select(L, 64, ub, k_sel, sink, recent)
            n = int(cnt[b, h])
            got = idx[b, h, :n]
            assert n == len(want), (b, h, n, len(want))
            assert np.all(np.diff(got) > 0)
            se, rb = oracle.forced_range(L, 64, sink, recent)
            for j in set(got.tolist()) ^ set(want.tolist()):
                assert se <= j < rb
                assert abs(ub[j] - kth) <= TIE_REL * max(abs(kth), mag[j]), (b, h, j)


@pytest.mark.parametrize("dtype", [kvd.F16, kvd.INT8, kvd.Q4_0])
@pytest.mark.parametrize("G", [2, 4, 8])
def test_per_head_select_and_decode_match_oracle(dtype, G):
    B, Hkv, L = 2, 2, 64 * 41 + 13
    gc, oc, q = _case(dtype, B, Hkv, G, L, 600 + G)
    ws = kvd.make_workspace(gc, Hkv * G)
    k_sel, sink, recent = 7, 4, 100
    sel_idx, sel_cnt = _select(gc, q, k_sel, sink, recent, ws)
    max_sel = kvd.selected_count(L, k_sel, sink, recent)
    out = torch.full((B, Hkv * G, 128), float("nan"), device=dev())
    kvd.decode_attn_per_head(gc, q, scale_for(), sel_idx, sel_cnt, max_sel, out, ws)
    torch.cuda.synchronize()
    q_np = q.cpu().numpy()
    _check_lists(sel_idx, sel_cnt, oc, q_np, k_sel, sink, recent, G)
    idx, cnt = sel_idx.cpu().numpy(), sel_cnt.cpu().numpy()
    # the heads of a group do choose differently (else the ablation shows nothing)
    assert any(set(idx[0, 0, :cnt[0, 0]]) != set(idx[0, h, :cnt[0, h]]) for h in range(1, G))
    for b in range(B):
        for h in range(Hkv * G):
            g = h // G
            sel = idx[b, h, :cnt[b, h]]
            if dtype == kvd.F16:
                ref = oracle.attend_f16(q_np[b, h], oc.K[b, g], oc.V[b, g], L, 64, scale_for(),
                                        sel=sel)
            else:
                qc, qs = oracle.quantize_row(q_np[b, h])
                if dtype == kvd.INT8:
                    ref = oracle.attend_int8(qc, qs, oc.K[b, g], oc.V[b, g], oc.ks[b, g],
                                             oc.vs[b, g], L, 64, scale_for(), sel=sel)
                else:
                    ref, _ = oracle.attend_q4_0(qc, qs, oc.K[b, g], oc.V[b, g], oc.kd[b, g],
                                                oc.vd[b, g], L, 64, scale_for(), sel=sel)
            assert_outputs(out[b, h:h + 1], ref[None], dtype, f"per-head {dtype} b{b} h{h}")
    assert gc.device_status() == 0


def test_one_head_per_group_is_the_shared_path():
    B, Hkv, G, L = 1, 8, 1, 5000
    gc, oc, q = _case(kvd.INT8, B, Hkv, G, L, 650)
    ws = kvd.make_workspace(gc, Hkv)
    nbmax = gc.max_seq // 64
    a_idx = torch.zeros((B, Hkv, nbmax), dtype=torch.int32, device=dev())
    a_cnt = torch.zeros((B, Hkv), dtype=torch.int32, device=dev())
    kvd.select_blocks(gc, q, 9, 4, 64, a_idx, a_cnt, ws)
    b_idx, b_cnt = _select(gc, q, 9, 4, 64, ws)
    max_sel = kvd.selected_count(L, 9, 4, 64)
    a = torch.empty((B, Hkv, 128), device=dev())
    b_ = torch.empty_like(a)
    kvd.decode_attn(gc, q, scale_for(), a_idx, a_cnt, max_sel, a, ws)
    kvd.decode_attn_per_head(gc, q, scale_for(), b_idx, b_cnt, max_sel, b_, ws)
    torch.cuda.synchronize()
    assert torch.equal(a_cnt, b_cnt)
    for g in range(Hkv):
        n = int(a_cnt[0, g])
        assert torch.equal(a_idx[0, g, :n], b_idx[0, g, :n])
    assert torch.equal(a, b_)


@pytest.mark.parametrize("k_sel", [0, 10 ** 6])
def test_nothing_to_rank_fills_every_head(k_sel):
    # K_SEL 0 or at least the candidate count: every head gets the forced (or
    # every) block, through the fill path
    B, Hkv, G, L = 1, 2, 4, 64 * 20 + 5
    gc, oc, q = _case(kvd.F16, B, Hkv, G, L, 660)
    ws = kvd.make_workspace(gc, Hkv * G)
    sel_idx, sel_cnt = _select(gc, q, k_sel, 64, 64, ws)
    torch.cuda.synchronize()
    want, _ = oracle.select(L, 64, np.zeros((L + 63) // 64), k_sel, 64, 64)
    for h in range(Hkv * G):
        assert int(sel_cnt[0, h]) == len(want)
        assert sel_idx[0, h, :len(want)].cpu().tolist() == want.tolist()
