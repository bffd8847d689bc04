"""The decode workloads at full size, run the way the benchmark runs them
(one whole decode step through the C ABI: append the step's token, select,
attend), checked against the oracle on sampled (sequence, KV head) problems
and, for the small ones, everywhere.

Per sampled problem: cache rows (codes, scales) of the needles, of random
positions and of the step's token bit-exact; every block bound equal; the
selection identical up to the tie window; the G query heads' outputs within
the stated tolerance and within 1e-4 of the oracle's attention over the
GPU's own list (so a legitimate tie swap never leaves a problem unchecked;
every sampled problem is compared, and the count is asserted).  Needle
recall: every planted needle's block is selected in the 32K and 128K
workloads; at 1M (random-walk keys) the recall is reported, and a needle the
GPU drops must be dropped by the oracle's selection too.
"""
import numpy as np
import pytest
import torch

import long_context_decode_kv_gb300 as kvd
import oracle
from long_context_decode_kv_gb300 import synth
from gpu_util import (TOL, assert_outputs, check_selection, dev, oracle_attend_list,
                      rel_l2_rows)

pytestmark = pytest.mark.gpu


def _build(w):
    q, k, v, needles = synth.make_workload(w, device=dev())
    gc = kvd.KVCache(w.dtype, w.B, w.Hkv, w.L + 64, device=dev())
    kvd.kv_append(gc, k, v)
    return q, k, v, needles, gc


def _oracle_problem(w, k, v, b, g, kn, vn):
    oc = oracle.OracleCache(w.dtype, 1, 1, w.D, w.L + 64, 64)
    oc.append(k[b:b + 1, :, g:g + 1].contiguous().cpu().numpy(),
              v[b:b + 1, :, g:g + 1].contiguous().cpu().numpy())
    oc.append(kn[b:b + 1, :, g:g + 1].cpu().numpy(), vn[b:b + 1, :, g:g + 1].cpu().numpy())
    return oc


def _check_rows(gc, oc, b, g, rows):
    rows = np.asarray(sorted(set(int(r) for r in rows)))
    if gc.dtype == kvd.INT8:
        assert np.array_equal(gc.k[b, g, rows].cpu().numpy(), oc.K[0, 0, rows])
        assert np.array_equal(gc.v[b, g, rows].cpu().numpy(), oc.V[0, 0, rows])
        assert np.array_equal(gc.k_scale[b, g, rows].cpu().numpy().view(np.uint32),
                              oc.ks[0, 0, rows].view(np.uint32))
        assert np.array_equal(gc.v_scale[b, g, rows].cpu().numpy().view(np.uint32),
                              oc.vs[0, 0, rows].view(np.uint32))
    else:
        assert np.array_equal(gc.k[b, g, rows].cpu().view(torch.int16).numpy(),
                              oc.K[0, 0, rows].view(np.int16))
    nb = (oc.len + 63) // 64
    assert np.array_equal(gc.kmin[b, g, :nb].cpu().float().numpy(),
                          oc.kmin[0, 0, :nb].astype(np.float32))
    assert np.array_equal(gc.kmax[b, g, :nb].cpu().float().numpy(),
                          oc.kmax[0, 0, :nb].astype(np.float32))


def _run(w, samples, dense_too=False):
    q, k, v, needles, gc = _build(w)
    kn, vn = synth.make_step_token(w, 0, device=dev())
    ws = kvd.make_workspace(gc, w.H)
    nbmax = gc.max_seq // 64
    sel_idx = torch.zeros((w.B, w.Hkv, nbmax), dtype=torch.int32, device=dev())
    sel_cnt = torch.zeros((w.B, w.Hkv), dtype=torch.int32, device=dev())
    out = torch.empty(w.B, w.H, w.D, device=dev())
    kvd.decode_step(gc, q, kn, vn, w.scale, w.k_sel, w.sink_tokens, w.recent_tokens, out, ws,
                    sel_idx=sel_idx, sel_cnt=sel_cnt)
    dense = None
    if dense_too:
        dense = torch.empty_like(out)
        kvd.decode_attn_dense(gc, q, w.scale, dense, ws)
    torch.cuda.synchronize()
    assert gc.device_status() == 0
    L1 = w.L + 1
    assert torch.all(sel_cnt == kvd.selected_count(L1, w.k_sel, w.sink_tokens, w.recent_tokens))
    idx, cnt = sel_idx.cpu().numpy(), sel_cnt.cpu().numpy()
    missed = {(b, g): [int(p) for p in needles[b, g].cpu().tolist()
                       if int(p) // 64 not in set(idx[b, g, :cnt[b, g]].tolist())]
              for b in range(w.B) for g in range(w.Hkv)}
    rng = np.random.default_rng(w.seed)
    qn = q.cpu().numpy()
    G = w.G
    worst = 0.0
    compared = 0
    for b, g in samples:
        oc = _oracle_problem(w, k, v, b, g, kn, vn)
        rows = list(needles[b, g].cpu().numpy()) + list(rng.integers(0, w.L, 64)) + [w.L]
        _check_rows(gc, oc, b, g, rows)
        qg = qn[b:b + 1, g * G:(g + 1) * G]
        swaps = check_selection(sel_idx[b:b + 1, g:g + 1], sel_cnt[b:b + 1, g:g + 1], oc, qg,
                                w.k_sel, w.sink_tokens, w.recent_tokens, G)
        _, o_idx, o_cnt = oc.decode(qg, w.scale, k_sel=w.k_sel, sink_tokens=w.sink_tokens,
                                    recent_tokens=w.recent_tokens)
        # a needle the GPU dropped must be dropped by the oracle's selection too
        o_sel = set(o_idx[0, 0, :o_cnt[0, 0]].tolist())
        assert all(p // 64 not in o_sel for p in missed[(b, g)]), (b, g, missed[(b, g)])
        # the oracle attends the GPU's own list: identical to the oracle's
        # selection, or different only inside the tie window (checked above)
        ref = oracle_attend_list(oc, qg[0], 0, 0, idx[b, g, :cnt[b, g]], w.scale)
        err = assert_outputs(out[b, g * G:(g + 1) * G], ref, w.dtype, f"{w.name} b{b} g{g}")
        worst = max(worst, err)
        compared += 1
        line = f"{w.name} b{b} g{g}: sparse rel-L2 {err:.2e}, tie swaps {swaps}"
        if dense is not None:
            dref, _, _ = oc.decode(qg, w.scale, dense=True)
            derr = assert_outputs(dense[b, g * G:(g + 1) * G], dref[0], w.dtype,
                                  f"{w.name} dense b{b} g{g}")
            line += f", dense rel-L2 {derr:.2e}"
        print(line)
    assert compared == len(samples)
    n_missed = sum(len(m) for m in missed.values())
    recall = 1.0 - n_missed / max(1, w.B * w.Hkv * w.n_needles)
    print(f"{w.name}: needle recall {recall:.4f}, worst sampled rel-L2 {worst:.2e}")
    return recall


def test_tiny_512_f16_everywhere():
    w = synth.TINY
    q, k, v, _, gc = _build(w)
    oc = oracle.OracleCache(w.dtype, w.B, w.Hkv, w.D, w.L + 64, 64)
    oc.append(k.cpu().numpy(), v.cpu().numpy())
    ws = kvd.make_workspace(gc, w.H)
    nbmax = gc.max_seq // 64
    for k_sel in (w.k_sel, 10 ** 6):
        sel_idx = torch.zeros((w.B, w.Hkv, nbmax), dtype=torch.int32, device=dev())
        sel_cnt = torch.zeros((w.B, w.Hkv), dtype=torch.int32, device=dev())
        kvd.select_blocks(gc, q, k_sel, w.sink_tokens, w.recent_tokens, sel_idx, sel_cnt, ws)
        out = torch.empty(w.B, w.H, w.D, device=dev())
        kvd.decode_attn(gc, q, w.scale, sel_idx, sel_cnt, w.NB, out, ws)
        torch.cuda.synchronize()
        qn = q.cpu().numpy()
        check_selection(sel_idx, sel_cnt, oc, qn, k_sel, w.sink_tokens, w.recent_tokens, w.G)
        _, _, cnt = oc.decode(qn, w.scale, k_sel=k_sel, sink_tokens=w.sink_tokens,
                              recent_tokens=w.recent_tokens)
        assert int(cnt[0, 0]) == (6 if k_sel == w.k_sel else 8)
        idx, gcnt = sel_idx.cpu().numpy(), sel_cnt.cpu().numpy()
        for g in range(w.Hkv):
            ref = oracle_attend_list(oc, qn[0, g * w.G:(g + 1) * w.G], 0, g,
                                     idx[0, g, :gcnt[0, g]], w.scale)
            assert_outputs(out[0, g * w.G:(g + 1) * w.G], ref, w.dtype,
                           f"tiny k_sel={k_sel} g{g}")
    dense = torch.empty(w.B, w.H, w.D, device=dev())
    kvd.decode_attn_dense(gc, q, w.scale, dense, ws)
    torch.cuda.synchronize()
    ref, _, _ = oc.decode(q.cpu().numpy(), w.scale, dense=True)
    assert_outputs(dense, ref, w.dtype, "tiny dense")


@pytest.mark.parametrize("w", synth.INT8_DENSE, ids=lambda w: w.name)
def test_int8_dense_everywhere(w):
    q, k, v, _, gc = _build(w)
    oc = oracle.OracleCache(w.dtype, w.B, w.Hkv, w.D, w.L + 64, 64)
    oc.append(k.cpu().numpy(), v.cpu().numpy())
    ws = kvd.make_workspace(gc, w.H)
    out = torch.empty(w.B, w.H, w.D, device=dev())
    kvd.decode_attn_dense(gc, q, w.scale, out, ws)
    torch.cuda.synchronize()
    # codes and scales of the whole cache
    assert np.array_equal(gc.k[:, :, :w.L].cpu().numpy(), oc.K[:, :, :w.L])
    assert np.array_equal(gc.v_scale[:, :, :w.L].cpu().numpy().view(np.uint32),
                          oc.vs[:, :, :w.L].view(np.uint32))
    ref, _, _ = oc.decode(q.cpu().numpy(), w.scale, dense=True)
    assert_outputs(out, ref, w.dtype, w.name)
    # cpu-attn "Correctness": against fp32 attention with the unquantized query on
    # the dequantized cache (query rounding included): median of the heads
    errs = []
    qn = q.cpu().numpy()
    for h in range(w.H):
        f = oracle.attend_dequant(qn[0, h], oc.K[0, h], oc.V[0, h], oc.ks[0, h], oc.vs[0, h],
                                  w.L, 64, w.scale)
        errs.append(rel_l2_rows(out[0, h:h + 1], f[None])[0])
    assert np.median(errs) < TOL[kvd.INT8]


def test_qwen3_gqa_32k_f16_every_problem():
    w = synth.QWEN3_32K
    assert _run(w, [(0, g) for g in range(w.Hkv)], dense_too=True) == 1.0


def test_ctx128k_batch8_int8_sampled():
    # ten problems over all eight sequences and all eight KV heads
    w = synth.CTX128K_B8
    samples = [(0, 0), (7, 7)] + [(b, (3 * b + 1) % w.Hkv) for b in range(w.B)]
    assert _run(w, samples, dense_too=True) == 1.0


def test_ctx1m_int8_sampled():
    # With the random-walk drift of this workload (per-channel offsets reach
    # ~10 sigma-units by 1M tokens), the Quest bound of late blocks is driven
    # by the drift term q.w and can pass that of an early needle's block: the
    # needle recall of top-1024 is below 1 here, for the oracle's selection
    # as much as for the GPU's (checked on the sampled problems).
    w = synth.CTX1M
    recall = _run(w, [(0, g) for g in range(w.Hkv)], dense_too=True)
    assert recall > 0.5
