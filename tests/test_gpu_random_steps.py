"""Seeded random decode steps against the oracle.

Each case draws a cache type, a batch, KV heads, a group size, per-sequence
lengths (or one length), a budget (K_SEL, sink, recent, or the dense arm) and
whether the cache keeps block means, fills the cache through per-sequence
views, runs three kvd_decode_step calls, and compares every (sequence, KV
head) with an oracle cache of that sequence:

  * selected lists: identical to the oracle's top-K on that sequence's own
    length up to the tie window;
  * outputs: within the cache type's bar and 1e-4 of the oracle's attention
    on the GPU's lists;
  * block means (when kept): within one f16 step of the oracle's.
"""
import numpy as np
import pytest
import torch

import long_context_decode_kv_gb300 as kvd
import oracle
from gpu_util import TIE_REL, assert_outputs, dev, scale_for, seeded

pytestmark = pytest.mark.gpu
DTYPES = [kvd.F16, kvd.INT8, kvd.Q8_0, kvd.Q4_0]


def _draw(seed):
    rng = np.random.default_rng(seed)
    dtype = DTYPES[seed % 4]
    B = int(rng.integers(1, 4))
    Hkv = int(rng.choice([1, 2, 4]))
    G = int(rng.choice([1, 2, 4, 8]))
    varlen = bool(rng.integers(0, 2))
    if varlen:
        lens = [int(x) for x in rng.integers(0, 5000, B)]
    else:
        lens = [int(rng.integers(1, 5000))] * B
    dense = rng.random() < 0.2
    k_sel = -1 if dense else int(rng.integers(0, 40))
    sink = int(rng.choice([0, 1, 4, 64, 100]))
    recent = int(rng.choice([0, 1, 64, 300]))
    moments = bool(rng.integers(0, 2))
    return dtype, B, Hkv, G, lens, k_sel, sink, recent, moments, varlen


def _head_ref(dtype, oc, qh, g, sel):
    L = oc.len
    if dtype == kvd.F16:
        return oracle.attend_f16(qh, oc.K[0, g], oc.V[0, g], L, 64, scale_for(), sel=sel)
    qc, qs = oracle.quantize_row(qh)
    if dtype == kvd.INT8:
        return oracle.attend_int8(qc, qs, oc.K[0, g], oc.V[0, g], oc.ks[0, g], oc.vs[0, g], L,
                                  64, scale_for(), sel=sel)
    att = oracle.attend_q8_0 if dtype == kvd.Q8_0 else oracle.attend_q4_0
    return att(qc, qs, oc.K[0, g], oc.V[0, g], oc.kd[0, g], oc.vd[0, g], L, 64, scale_for(),
               sel=sel)[0]


@pytest.mark.parametrize("seed", range(16))
def test_random_steps(seed):
    dtype, B, Hkv, G, lens, k_sel, sink, recent, moments, varlen = _draw(seed)
    max_seq = (max(lens) + 3 + 63) // 64 * 64 + 64
    gc = kvd.KVCache(dtype, B, Hkv, max_seq, device=dev(), moments=moments)
    ocs = []
    for b, L in enumerate(lens):
        oc = oracle.OracleCache(dtype, 1, Hkv, 128, max_seq, 64)
        if L:
            k = seeded((1, L, Hkv, 128), 1000 * seed + 3 * b, scale=1.5)
            v = seeded((1, L, Hkv, 128), 1000 * seed + 3 * b + 1)
            kvd.kv_append(gc.view(b), k, v)
            oc.append(k.cpu().numpy(), v.cpu().numpy())
        ocs.append(oc)
    lens_t = torch.tensor(lens, dtype=torch.int32, device=dev())
    if varlen:
        gc.set_seq_lens(lens_t)
    gc.len = max(lens)
    ws = kvd.make_workspace(gc, Hkv * G)
    nbmax = gc.max_seq // 64
    sel_idx = torch.zeros((B, Hkv, nbmax), dtype=torch.int32, device=dev())
    sel_cnt = torch.zeros((B, Hkv), dtype=torch.int32, device=dev())
    out = torch.empty((B, Hkv * G, 128), device=dev())
    what = f"seed {seed}: {dtype} B{B} Hkv{Hkv} G{G} lens{lens} k{k_sel} s{sink} r{recent}"
    for step in range(3):
        q = seeded((B, Hkv * G, 128), 1000 * seed + 500 + step, scale=2.0, dtype=torch.float32)
        kn = seeded((B, 1, Hkv, 128), 1000 * seed + 600 + step)
        vn = seeded((B, 1, Hkv, 128), 1000 * seed + 700 + step)
        kvd.decode_step(gc, q, kn, vn, scale_for(), k_sel, sink, recent, out, ws, sel_idx,
                        sel_cnt)
        if varlen:
            lens_t += 1
        torch.cuda.synchronize()
        assert gc.device_status() == 0, what
        q_np = q.cpu().numpy()
        idx, cnt = sel_idx.cpu().numpy(), sel_cnt.cpu().numpy()
        for b, oc in enumerate(ocs):
            oc.append(kn[b:b + 1].cpu().numpy(), vn[b:b + 1].cpu().numpy())
            L = oc.len
            nb = (L + 63) // 64
            for g in range(Hkv):
                sel = None
                if k_sel >= 0:
                    qg = q_np[b, g * G:(g + 1) * G]
                    ub, _, mag = oracle.block_scores(qg, oc.kmin[0, g, :nb], oc.kmax[0, g, :nb])
                    want, kth = oracle.select(L, 64, ub, k_sel, sink, recent)
                    n = int(cnt[b, g])
                    sel = idx[b, g, :n]
                    assert n == len(want), (what, step, b, g)
                    se, rb = oracle.forced_range(L, 64, sink, recent)
                    for j in set(sel.tolist()) ^ set(want.tolist()):
                        assert se <= j < rb, (what, step, b, g, j)
                        assert abs(ub[j] - kth) <= TIE_REL * max(abs(kth), mag[j]), what
                ref = np.stack([_head_ref(dtype, oc, q_np[b, g * G + h], g, sel)
                                for h in range(G)])
                assert_outputs(out[b, g * G:(g + 1) * G], ref, dtype, f"{what} step {step}")
    if moments:
        for b, oc in enumerate(ocs):
            nb = (oc.len + 63) // 64
            got = gc.moments[b, :, :nb].cpu().numpy().astype(np.float64)
            for g in range(Hkv):
                mK, mV = oc.moments(0, g)
                for i, want in enumerate((mK, mV)):
                    step16 = np.spacing(np.abs(want)).astype(np.float64)
                    assert np.all(np.abs(got[g, :, i] - want) <= step16), (what, b, g, i)
