"""GPU split-KV decode attention (sparse over a selection, and dense) vs the oracle.

Bar: relative L2 per (sequence, query head) within 2e-3 (f16) / 8e-3 (int8)
and within 1e-4; int8 dots, query codes and scales bit-exact.
"""
import os

import numpy as np
import pytest
import torch

import long_context_decode_kv_gb300 as kvd
import oracle
from gpu_util import assert_outputs, dev, make_pair, scale_for, seeded

pytestmark = pytest.mark.gpu


def _q(B, H, seed, scale=1.0):
    return seeded((B, H, 128), seed, scale=scale, dtype=torch.float32)


def _dense(gc, q, scale, ws=None):
    ws = kvd.make_workspace(gc, q.shape[1]) if ws is None else ws
    out = torch.full((q.shape[0], q.shape[1], 128), float("nan"), device=dev())
    kvd.decode_attn_dense(gc, q, scale, out, ws)
    torch.cuda.synchronize()
    return out


def _sparse(gc, q, scale, sel_idx, sel_cnt, max_sel, ws=None):
    ws = kvd.make_workspace(gc, q.shape[1]) if ws is None else ws
    out = torch.full((q.shape[0], q.shape[1], 128), float("nan"), device=dev())
    kvd.decode_attn(gc, q, scale, sel_idx, sel_cnt, max_sel, out, ws)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("dtype", [kvd.F16, kvd.INT8, kvd.Q8_0, kvd.Q4_0])
@pytest.mark.parametrize("B,Hkv,G,L", [
    (1, 1, 1, 1), (1, 2, 1, 63), (1, 8, 1, 512), (2, 2, 4, 1000), (1, 8, 4, 4097),
    (1, 2, 2, 777), (1, 1, 8, 2000), (1, 1, 16, 300), (40, 8, 4, 200), (3, 1, 4, 20000),
])
def test_dense_matches_oracle(dtype, B, Hkv, G, L):
    k = seeded((B, L, Hkv, 128), 61 + L)
    v = seeded((B, L, Hkv, 128), 62 + L)
    gc, oc = make_pair(dtype, k, v)
    q = _q(B, Hkv * G, 63)
    out = _dense(gc, q, scale_for())
    ref, _, _ = oc.decode(q.cpu().numpy(), scale_for(), dense=True)
    assert_outputs(out, ref, dtype, f"dense {dtype} B{B} Hkv{Hkv} G{G} L{L}")


@pytest.mark.parametrize("dtype", [kvd.F16, kvd.INT8, kvd.Q8_0, kvd.Q4_0])
@pytest.mark.parametrize("L,k_sel,sink,recent", [
    (512, 4, 4, 64), (1000, 3, 0, 1), (5000, 20, 4, 256), (20000, 50, 64, 1000),
])
def test_sparse_with_oracle_selection(dtype, L, k_sel, sink, recent):
    B, Hkv, G = 2, 2, 4
    k = seeded((B, L, Hkv, 128), 71 + L, scale=1.5)
    v = seeded((B, L, Hkv, 128), 72 + L)
    gc, oc = make_pair(dtype, k, v)
    q = _q(B, Hkv * G, 73, scale=2.0)
    ref, o_idx, o_cnt = oc.decode(q.cpu().numpy(), scale_for(), k_sel=k_sel, sink_tokens=sink,
                                  recent_tokens=recent)
    sel_idx = torch.from_numpy(o_idx).to(dev())
    sel_cnt = torch.from_numpy(o_cnt).to(dev())
    out = _sparse(gc, q, scale_for(), sel_idx, sel_cnt, int(o_cnt.max()))
    assert_outputs(out, ref, dtype, f"sparse {dtype} L{L}")


@pytest.mark.parametrize("dtype", [kvd.INT8, kvd.Q8_0, kvd.Q4_0])
@pytest.mark.parametrize("B,Hkv", [(1, 8), (10, 4)])
def test_sparse_both_tiles(dtype, B, Hkv):
    # few problems take the wide tile (one CTA per SM, four consumer groups),
    # many take two CTAs per SM: both against the oracle
    L, G = 3000, 4
    k = seeded((B, L, Hkv, 128), 91, scale=1.5)
    v = seeded((B, L, Hkv, 128), 92)
    gc, oc = make_pair(dtype, k, v)
    q = _q(B, Hkv * G, 93, scale=2.0)
    ref, o_idx, o_cnt = oc.decode(q.cpu().numpy(), scale_for(), k_sel=9, sink_tokens=4,
                                  recent_tokens=128)
    sel_idx = torch.from_numpy(o_idx).to(dev())
    sel_cnt = torch.from_numpy(o_cnt).to(dev())
    out = _sparse(gc, q, scale_for(), sel_idx, sel_cnt, int(o_cnt.max()))
    assert_outputs(out, ref, dtype, f"sparse {dtype} B{B} Hkv{Hkv}")


@pytest.mark.parametrize("dtype", [kvd.F16, kvd.INT8, kvd.Q8_0, kvd.Q4_0])
def test_select_all_equals_dense(dtype):
    # gate ladder plumbing anchor: K_SEL = n_blocks => sparse == dense
    B, Hkv, G, L = 2, 4, 4, 3333
    k = seeded((B, L, Hkv, 128), 81)
    v = seeded((B, L, Hkv, 128), 82)
    gc, oc = make_pair(dtype, k, v)
    q = _q(B, Hkv * G, 83)
    ws = kvd.make_workspace(gc, Hkv * G)
    sel_idx = torch.zeros((B, Hkv, gc.max_seq // 64), dtype=torch.int32, device=dev())
    sel_cnt = torch.zeros((B, Hkv), dtype=torch.int32, device=dev())
    kvd.select_blocks(gc, q, 10 ** 6, 0, 0, sel_idx, sel_cnt, ws)
    nb = (L + 63) // 64
    sp = _sparse(gc, q, scale_for(), sel_idx, sel_cnt, nb, ws)
    de = _dense(gc, q, scale_for(), ws)
    assert torch.all(sel_cnt == nb)
    assert torch.allclose(sp, de, rtol=1e-6, atol=1e-7)
    ref, _, _ = oc.decode(q.cpu().numpy(), scale_for(), dense=True)
    assert_outputs(sp, ref, dtype, "select-all")


@pytest.mark.parametrize("dtype", [kvd.F16, kvd.INT8])
def test_uniform_logits_give_mean_of_v(dtype):
    B, Hkv, G, L = 1, 2, 4, 1500
    k = seeded((B, L, Hkv, 128), 91)
    v = seeded((B, L, Hkv, 128), 92)
    gc, oc = make_pair(dtype, k, v)
    q = torch.zeros(B, Hkv * G, 128, device=dev())
    out = _dense(gc, q, scale_for())
    for g in range(Hkv):
        if dtype == kvd.F16:
            mean = v[0, :, g].double().mean(0).cpu().numpy()
        else:
            mean = (oc.vs[0, g, :L, None].astype(np.float64) * oc.V[0, g, :L]).mean(0)
        for h in range(G):
            got = out[0, g * G + h].double().cpu().numpy()
            assert np.linalg.norm(got - mean) <= 1e-5 * np.linalg.norm(mean)


def test_int8_dots_and_query_codes_bit_exact():
    B, Hkv, G, L = 2, 2, 4, 700
    k = seeded((B, L, Hkv, 128), 101, scale=3.0)
    gc, oc = make_pair(kvd.INT8, k, k)
    q = _q(B, Hkv * G, 102)
    q[0, 0, :4] = torch.tensor([float.fromhex("0x1.8p-139"), -float.fromhex("0x1.8p-139"),
                                float.fromhex("0x1p-140"), 0.0])
    q[0, 0, 4:] = 0.0          # golden subnormal query row (R1 clamp case)
    q[1, 3] = 0.0              # zero row: scale 0, codes 0
    dots = torch.zeros(B, Hkv * G, L, dtype=torch.int32, device=dev())
    codes = torch.zeros(B, Hkv * G, 128, dtype=torch.int8, device=dev())
    scales = torch.zeros(B, Hkv * G, device=dev())
    kvd.debug_qk_int8(gc, q, dots, codes, scales)
    torch.cuda.synchronize()
    qn = q.cpu().numpy()
    assert codes[0, 0, :4].cpu().tolist() == [127, -127, 43, 0]
    for b in range(B):
        for h in range(Hkv * G):
            c, s = oracle.quantize_row(qn[b, h])
            assert np.array_equal(codes[b, h].cpu().numpy(), c)
            assert scales[b, h].cpu().numpy().view(np.uint32) == np.float32(s).view(np.uint32)
            want = oracle.qk_int8(c, oc.K[b, h // G, :L])
            assert np.array_equal(dots[b, h].cpu().numpy().astype(np.int64), want)


def test_empty_selection_and_bad_ids():
    B, Hkv, G, L = 1, 2, 4, 640
    k = seeded((B, L, Hkv, 128), 111)
    gc, oc = make_pair(kvd.F16, k, k)
    q = _q(B, Hkv * G, 112)
    sel_idx = torch.zeros((B, Hkv, gc.max_seq // 64), dtype=torch.int32, device=dev())
    sel_cnt = torch.zeros((B, Hkv), dtype=torch.int32, device=dev())
    out = _sparse(gc, q, scale_for(), sel_idx, sel_cnt, 1)
    assert torch.all(out == 0)
    # ids outside [0, NB) are skipped and reported; the valid ones still count
    sel_idx[0, :, 0] = 3
    sel_idx[0, :, 1] = 10 ** 6
    sel_idx[0, :, 2] = -5
    sel_cnt[:] = 3
    out = _sparse(gc, q, scale_for(), sel_idx, sel_cnt, 3)
    assert gc.device_status() == 1  # KVD_ERR_INVALID
    gc.status.zero_()
    ref, _, _ = oc.decode(q.cpu().numpy(), scale_for(), k_sel=0, sink_tokens=0, recent_tokens=0)
    for g in range(Hkv):
        want = [oracle.attend_f16(q.cpu().numpy()[0, g * G + h], oc.K[0, g], oc.V[0, g], L, 64,
                                  scale_for(), sel=np.array([3], np.int32)) for h in range(G)]
        assert_outputs(out[0, g * G:(g + 1) * G], np.stack(want), kvd.F16, "bad ids")


@pytest.mark.parametrize("dtype", [kvd.F16, kvd.INT8])
def test_repeated_calls_identical(dtype):
    # split partials and the arrival counters are reused call after call
    B, Hkv, G, L = 1, 8, 4, 30000
    k = seeded((B, L, Hkv, 128), 121)
    v = seeded((B, L, Hkv, 128), 122)
    gc, _ = make_pair(dtype, k, v)
    q = _q(B, Hkv * G, 123)
    ws = kvd.make_workspace(gc, Hkv * G)
    outs = [_dense(gc, q, scale_for(), ws) for _ in range(4)]
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


def test_large_logits_stay_finite():
    # a strongly peaked softmax (needle keys) must not overflow
    B, Hkv, G, L = 1, 1, 4, 2048
    k = seeded((B, L, Hkv, 128), 131)
    q = _q(B, Hkv * G, 132)
    qd = q[0].mean(0)
    k[0, 1234, 0] = (qd / qd.norm() * 40).half()
    v = seeded((B, L, Hkv, 128), 133)
    for dtype in (kvd.F16, kvd.INT8):
        gc, oc = make_pair(dtype, k, v)
        out = _dense(gc, q, 1.0)
        ref, _, _ = oc.decode(q.cpu().numpy(), 1.0, dense=True)
        assert_outputs(out, ref, dtype, "peaked")
