"""GPU Quest bounds and block selection vs the oracle.

Bar: bounds within f32 rounding of the fp64 bound; selected sets identical
except inside the tie window around the K-th bound (see gpu_util).
"""
import numpy as np
import pytest
import torch

import long_context_decode_kv_gb300 as kvd
import oracle
from gpu_util import TIE_REL, check_selection, dev, make_pair, oracle_scores, seeded

pytestmark = pytest.mark.gpu


def _q(B, H, seed, scale=1.0):
    return seeded((B, H, 128), seed, scale=scale, dtype=torch.float32)


@pytest.mark.parametrize("G", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("dtype", [kvd.F16, kvd.INT8, kvd.Q8_0, kvd.Q4_0])
def test_scores_match_oracle(G, dtype):
    B, Hkv, L = 2, 2, 1000
    k = seeded((B, L, Hkv, 128), 31) + 0.5
    v = seeded((B, L, Hkv, 128), 32)
    gc, oc = make_pair(dtype, k, v)
    q = _q(B, Hkv * G, 33)
    nb = (L + 63) // 64
    ub = torch.empty(B, Hkv, nb, device=dev())
    kvd.debug_scores(gc, q, ub)
    torch.cuda.synchronize()
    qn = q.cpu().numpy()
    for b in range(B):
        for g in range(Hkv):
            want, _, mag = oracle_scores(oc, qn, b, g, G, L)
            got = ub[b, g].cpu().double().numpy()
            assert np.all(np.abs(got - want) <= 4e-6 * np.maximum(np.abs(want), mag) + 1e-30)


CASES = [
    # L, k_sel, sink, recent
    (512, 4, 4, 64),
    (512, 0, 4, 64),
    (512, 6, 4, 64),
    (512, 100, 0, 0),
    (500, 2, 65, 1),
    (1, 3, 0, 0),
    (130, 1, 0, 0),
    (5000, 17, 4, 256),
    (5000, 60, 0, 1),
    (20000, 77, 128, 640),
    # at most 512 candidates rank in one CTA; more go through the radix tail
    (32768, 100, 0, 0),     # 512 candidates
    (32769, 100, 0, 0),     # 513
    (40000, 300, 4, 256),
    (70000, 9, 0, 0),
]


@pytest.mark.parametrize("L,k_sel,sink,recent", CASES)
@pytest.mark.parametrize("G", [1, 4])
def test_select_matches_oracle(L, k_sel, sink, recent, G):
    B, Hkv = 2, 2
    k = seeded((B, L, Hkv, 128), 41 + L)
    v = seeded((B, L, Hkv, 128), 42)
    gc, oc = make_pair(kvd.F16, k, v)
    q = _q(B, Hkv * G, 43)
    ws = kvd.make_workspace(gc, Hkv * G)
    sel_idx = torch.full((B, Hkv, gc.max_seq // 64), -7, dtype=torch.int32, device=dev())
    sel_cnt = torch.full((B, Hkv), -7, dtype=torch.int32, device=dev())
    kvd.select_blocks(gc, q, k_sel, sink, recent, sel_idx, sel_cnt, ws)
    torch.cuda.synchronize()
    check_selection(sel_idx, sel_cnt, oc, q.cpu().numpy(), k_sel, sink, recent, G)
    assert np.all(sel_cnt.cpu().numpy() == kvd.selected_count(L, k_sel, sink, recent))


@pytest.mark.parametrize("nb", [40, 600])
def test_exact_ties_go_to_lower_index(nb):
    # every block identical => every bound equal (bit-identical f32 sums):
    # the top-K must be the lowest-index candidates (one-CTA and radix paths)
    B, Hkv, L, G = 1, 2, 64 * nb, 4
    row = seeded((1, 64, Hkv, 128), 5)
    k = row.repeat(1, nb, 1, 1).contiguous()
    v = seeded((B, L, Hkv, 128), 6)
    gc, oc = make_pair(kvd.F16, k, v)
    q = _q(B, Hkv * G, 7)
    ws = kvd.make_workspace(gc, Hkv * G)
    sel_idx = torch.zeros((B, Hkv, gc.max_seq // 64), dtype=torch.int32, device=dev())
    sel_cnt = torch.zeros((B, Hkv), dtype=torch.int32, device=dev())
    kvd.select_blocks(gc, q, 5, 1, 64, sel_idx, sel_cnt, ws)
    torch.cuda.synchronize()
    for g in range(Hkv):
        assert sel_idx[0, g, :sel_cnt[0, g]].cpu().tolist() == [0, 1, 2, 3, 4, 5, nb - 1]


def test_needle_blocks_survive_selection():
    # retrieval gate of the Quest page: every planted needle's block has to be
    # among the selected ones (needle keys lie along the group's query direction)
    from long_context_decode_kv_gb300 import synth
    w = synth.QWEN3_32K.with_(L=8192, k_sel=32)
    q, k, v, needles = synth.make_workload(w, device=dev())
    gc = kvd.KVCache(w.dtype, w.B, w.Hkv, w.L + 64, device=dev())
    kvd.kv_append(gc, k, v)
    ws = kvd.make_workspace(gc, w.H)
    sel_idx = torch.zeros((w.B, w.Hkv, gc.max_seq // 64), dtype=torch.int32, device=dev())
    sel_cnt = torch.zeros((w.B, w.Hkv), dtype=torch.int32, device=dev())
    kvd.select_blocks(gc, q, w.k_sel, w.sink_tokens, w.recent_tokens, sel_idx, sel_cnt, ws)
    torch.cuda.synchronize()
    for g in range(w.Hkv):
        sel = set(sel_idx[0, g, :sel_cnt[0, g]].cpu().tolist())
        for p in needles[0, g].cpu().tolist():
            assert p // 64 in sel


def test_select_repeatable_and_workspace_reuse():
    B, Hkv, L, G = 3, 2, 3000, 4
    k = seeded((B, L, Hkv, 128), 51)
    gc, oc = make_pair(kvd.INT8, k, k)
    q = _q(B, Hkv * G, 52)
    ws = kvd.make_workspace(gc, Hkv * G)
    outs = []
    for _ in range(3):
        sel_idx = torch.zeros((B, Hkv, gc.max_seq // 64), dtype=torch.int32, device=dev())
        sel_cnt = torch.zeros((B, Hkv), dtype=torch.int32, device=dev())
        kvd.select_blocks(gc, q, 9, 4, 64, sel_idx, sel_cnt, ws)
        outs.append((sel_idx.clone(), sel_cnt.clone()))
    torch.cuda.synchronize()
    for a, b in outs[1:]:
        assert torch.equal(a, outs[0][0]) and torch.equal(b, outs[0][1])
    check_selection(outs[0][0], outs[0][1], oc, q.cpu().numpy(), 9, 4, 64, G)


@pytest.mark.parametrize("B,Hkv,L,k_sel", [(24, 8, 3000, 9), (40, 8, 700, 3)])
def test_select_one_cta_per_problem(B, Hkv, L, k_sel):
    # more problems than SMs: each (sequence, KV head) is ranked by one CTA
    # (no barriers between CTAs); fewer problems split over several CTAs
    G = 4
    k = seeded((B, L, Hkv, 128), 61 + B)
    gc, oc = make_pair(kvd.F16, k, k)
    q = _q(B, Hkv * G, 62)
    ws = kvd.make_workspace(gc, Hkv * G)
    sel_idx = torch.full((B, Hkv, gc.max_seq // 64), -7, dtype=torch.int32, device=dev())
    sel_cnt = torch.full((B, Hkv), -7, dtype=torch.int32, device=dev())
    kvd.select_blocks(gc, q, k_sel, 4, 64, sel_idx, sel_cnt, ws)
    torch.cuda.synchronize()
    check_selection(sel_idx, sel_cnt, oc, q.cpu().numpy(), k_sel, 4, 64, G)


@pytest.mark.parametrize("nb,k_sel,G", [(36000, 700, 4), (49000, 2048, 8)])
def test_select_large_problem_keys_from_l2(nb, k_sel, G):
    # more candidates than the ranking CTA keeps in shared memory: it reads
    # the keys from L2.  Only bounds matter to the selection, so they are
    # written directly (kmin <= kmax per channel) instead of appending tokens.
    B, Hkv = 1, 1
    L = nb * 64 - 17
    gc = kvd.KVCache(kvd.INT8, B, Hkv, nb * 64, device=dev())
    a = seeded((B, Hkv, nb, 128), 81, scale=2.0)
    d = seeded((B, Hkv, nb, 128), 82).abs()
    gc.t["kbounds"][..., 0] = a
    gc.t["kbounds"][..., 1] = (a.float() + d.float()).half()
    gc.len = L
    q = _q(B, Hkv * G, 83)
    ws = kvd.make_workspace(gc, Hkv * G)
    sel_idx = torch.full((B, Hkv, nb), -7, dtype=torch.int32, device=dev())
    sel_cnt = torch.full((B, Hkv), -7, dtype=torch.int32, device=dev())
    kvd.select_blocks(gc, q, k_sel, 4, 256, sel_idx, sel_cnt, ws)
    torch.cuda.synchronize()
    kmin = gc.kmin[0, 0].cpu().numpy()
    kmax = gc.kmax[0, 0].cpu().numpy()
    ub, _, mag = oracle.block_scores(q[0].cpu().numpy(), kmin, kmax)
    want, kth = oracle.select(L, 64, ub, k_sel, 4, 256)
    n = int(sel_cnt[0, 0])
    got = sel_idx[0, 0, :n].cpu().numpy()
    assert n == len(want) and np.all(np.diff(got) > 0)
    for j in set(got.tolist()) ^ set(want.tolist()):
        assert abs(ub[j] - kth) <= TIE_REL * max(abs(kth), mag[j]), (j, ub[j], kth)


@pytest.mark.parametrize("cluster,nb", [(1000, 8192), (3000, 8192), (3000, 40000)])
def test_select_crowded_threshold_bin(cluster, nb):
    # Bounds are written so that each block's bound is one chosen f16 value
    # (q = e_0, channel 0's kmin = kmax = value, every other channel 0):
    # two outliers far above the rest, `cluster` blocks at 1 + 2^-10,
    # `cluster` at exactly 1, the rest at 0.5, in seeded order.  The K-th
    # pick lands among the exact ties at 1, which one bin of the first radix
    # digit holds together with the 1 + 2^-10 keys.  With 1000 per value the
    # bin's keys are collected and refined apart; with 3000 there are too
    # many to collect and the refinement re-reads every key (40000 blocks:
    # from L2).  Exact ties leave no freedom: the list must equal the
    # oracle's, lowest indices first.
    B, Hkv, G = 1, 1, 1
    L = nb * 64 - 17
    gc = kvd.KVCache(kvd.F16, B, Hkv, nb * 64, device=dev())
    cand = np.arange(1, nb - 5)  # clear of the sink block and the recent window
    rng = np.random.default_rng(91)
    perm = rng.permutation(cand)
    vals = np.full(nb, 0.5, np.float16)
    vals[perm[:2]] = 60000.0
    vals[perm[2:2 + cluster]] = 1.0 + 2.0 ** -10
    vals[perm[2 + cluster:2 + 2 * cluster]] = 1.0
    kb = torch.zeros((B, Hkv, nb, 128, 2), dtype=torch.float16)
    kb[0, 0, :, 0, 0] = torch.from_numpy(vals)
    kb[0, 0, :, 0, 1] = torch.from_numpy(vals)
    gc.t["kbounds"].copy_(kb.to(dev()))
    gc.len = L
    q = torch.zeros((B, Hkv * G, 128), dtype=torch.float32, device=dev())
    q[..., 0] = 1.0
    k_sel = 2 + cluster + cluster // 2
    ws = kvd.make_workspace(gc, Hkv * G)
    sel_idx = torch.full((B, Hkv, nb), -7, dtype=torch.int32, device=dev())
    sel_cnt = torch.full((B, Hkv), -7, dtype=torch.int32, device=dev())
    for _ in range(2):  # the second call runs on the scratch the first left
        kvd.select_blocks(gc, q, k_sel, 4, 256, sel_idx, sel_cnt, ws)
        torch.cuda.synchronize()
        ub, _, _ = oracle.block_scores(q[0].cpu().numpy(), gc.kmin[0, 0].cpu().numpy(),
                                       gc.kmax[0, 0].cpu().numpy())
        want, kth = oracle.select(L, 64, ub, k_sel, 4, 256)
        assert kth == 1.0
        n = int(sel_cnt[0, 0])
        assert sel_idx[0, 0, :n].cpu().numpy().tolist() == want.tolist()


@pytest.mark.parametrize("nb", [100, 531])
def test_select_bounds_of_both_signs(nb):
    # Each block's bound is one chosen f16 value (q = e_0, channel 0's kmin =
    # kmax = value): seeded normal values, so the keys of one problem span
    # negative and positive bounds (a key range of more than 2^31) and some
    # values repeat.  The bounds are exact, so the list must equal the
    # oracle's: the few-candidate ranking (100 blocks) and the radix tail (531).
    B, Hkv, G = 1, 1, 1
    L = nb * 64 - 17
    gc = kvd.KVCache(kvd.F16, B, Hkv, nb * 64, device=dev())
    rng = np.random.default_rng(97 + nb)
    vals = (rng.standard_normal(nb) * 4.0).astype(np.float16)
    vals[rng.integers(0, nb, 8)] = vals[3]  # ties
    kb = torch.zeros((B, Hkv, nb, 128, 2), dtype=torch.float16)
    kb[0, 0, :, 0, 0] = torch.from_numpy(vals)
    kb[0, 0, :, 0, 1] = torch.from_numpy(vals)
    gc.t["kbounds"].copy_(kb.to(dev()))
    gc.len = L
    q = torch.zeros((B, Hkv * G, 128), dtype=torch.float32, device=dev())
    q[..., 0] = 1.0
    ws = kvd.make_workspace(gc, Hkv * G)
    sel_idx = torch.full((B, Hkv, nb), -7, dtype=torch.int32, device=dev())
    sel_cnt = torch.full((B, Hkv), -7, dtype=torch.int32, device=dev())
    for k_sel in (1, nb // 3, nb - 20):
        kvd.select_blocks(gc, q, k_sel, 4, 256, sel_idx, sel_cnt, ws)
        torch.cuda.synchronize()
        ub, _, _ = oracle.block_scores(q[0].cpu().numpy(), gc.kmin[0, 0].cpu().numpy(),
                                       gc.kmax[0, 0].cpu().numpy())
        assert (ub < 0).any() and (ub > 0).any()
        want, _ = oracle.select(L, 64, ub, k_sel, 4, 256)
        n = int(sel_cnt[0, 0])
        assert sel_idx[0, 0, :n].cpu().numpy().tolist() == want.tolist(), k_sel
