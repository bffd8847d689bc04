"""Head dims other than 128 against the oracle (f16 and int8 caches).

"cpu-attn", Requirements and limits: a head dim that is a multiple of 16, at
most 1024.  The general kernels serve every such D but 128; the cases span
the smallest (16), dims that are not powers of two (80, 96, 144), and the
largest (1024), with group sizes 1 to 16; D = 64, 256 and 512 (the
warp-specialised decode kernel) with every group size it takes.

  * append: rows, scales and bounds bit-exact, across chunked appends that
    straddle blocks, from f16 and from f32 input;
  * selection: identical to the oracle's top-K up to the tie window;
  * decode: within the cache type's bar and 1e-4 of the oracle's attention
    on the GPU's lists, sparse and dense, and bit-identical on a repeat;
  * decode steps: three kvd_decode_step calls, sparse and dense, and the
    host-buffer step (pinned, pageable, mixed) equal to the device step.
"""
import numpy as np
import pytest
import torch

import long_context_decode_kv_gb300 as kvd
import oracle
from gpu_util import assert_outputs, check_selection, dev, make_pair, scale_for, seeded

pytestmark = pytest.mark.gpu
DTYPES = [kvd.F16, kvd.INT8]
CASES = [(16, 4), (64, 8), (80, 2), (96, 1), (144, 4), (256, 4), (1024, 16),
         # D = 64, 256 and 512 run the warp-specialised kernel: every head-group shape
         (64, 1), (64, 2), (64, 16), (256, 1), (256, 2), (256, 8), (256, 16), (512, 4),
         (512, 16)]


def _oracle_head(dtype, oc, qh, b, g, L, D, sel):
    if dtype == kvd.F16:
        return oracle.attend_f16(qh, oc.K[b, g], oc.V[b, g], L, 64, scale_for(D), sel=sel)
    qc, qs = oracle.quantize_row(qh)
    return oracle.attend_int8(qc, qs, oc.K[b, g], oc.V[b, g], oc.ks[b, g], oc.vs[b, g], L, 64,
                              scale_for(D), sel=sel)


def _check_outputs(dtype, gc, oc, q, out, G, D, sel_idx=None, sel_cnt=None, what=""):
    B, Hkv = gc.batch, gc.n_kv_heads
    q_np = q.cpu().numpy()
    idx = None if sel_idx is None else sel_idx.cpu().numpy()
    cnt = None if sel_cnt is None else sel_cnt.cpu().numpy()
    for b in range(B):
        for g in range(Hkv):
            sel = None if idx is None else idx[b, g, :int(cnt[b, g])]
            ref = np.stack([_oracle_head(dtype, oc, q_np[b, g * G + h], b, g, oc.len, D, sel)
                            for h in range(G)])
            assert_outputs(out[b, g * G:(g + 1) * G], ref, dtype, f"{what} b{b} g{g}")


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("D", [16, 80, 144, 1024])
def test_append_bit_exact(dtype, D):
    B, Hkv, L = 2, 3, 300
    k = seeded((B, L, Hkv, D), 11 + D, scale=2.0)
    v = seeded((B, L, Hkv, D), 12 + D)
    gc, oc = make_pair(dtype, k, v, max_seq=384, chunks=[1, 62, 3, 64, 100, 70])
    assert gc.device_status() == 0
    nb = (L + 63) // 64
    if dtype == kvd.F16:
        assert np.array_equal(gc.k[:, :, :L].cpu().numpy().view(np.uint16),
                              oc.K[:, :, :L].view(np.uint16))
        assert np.array_equal(gc.v[:, :, :L].cpu().numpy().view(np.uint16),
                              oc.V[:, :, :L].view(np.uint16))
    else:
        assert np.array_equal(gc.k[:, :, :L].cpu().numpy(), oc.K[:, :, :L])
        assert np.array_equal(gc.v[:, :, :L].cpu().numpy(), oc.V[:, :, :L])
        assert gc.k_scale[:, :, :L].cpu().numpy().tobytes() == oc.ks[:, :, :L].tobytes()
        assert gc.v_scale[:, :, :L].cpu().numpy().tobytes() == oc.vs[:, :, :L].tobytes()
    assert np.array_equal(gc.kmin[:, :, :nb].cpu().numpy().astype(np.float64),
                          oc.kmin[:, :, :nb].astype(np.float64))
    assert np.array_equal(gc.kmax[:, :, :nb].cpu().numpy().astype(np.float64),
                          oc.kmax[:, :, :nb].astype(np.float64))


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("D", [48, 256])
def test_append_f32_bit_exact(dtype, D):
    B, Hkv, L = 1, 2, 150
    k = seeded((B, L, Hkv, D), 21 + D, scale=3.0, dtype=torch.float32)
    v = seeded((B, L, Hkv, D), 22 + D, dtype=torch.float32)
    gc = kvd.KVCache(dtype, B, Hkv, 256, head_dim=D, device=dev())
    oc = oracle.OracleCache(dtype, B, Hkv, D, 256, 64)
    for s, e in ((0, 70), (70, 71), (71, 150)):
        kvd.kv_append_f32(gc, k[:, s:e].contiguous(), v[:, s:e].contiguous())
        oc.append_f32(k[:, s:e].cpu().numpy(), v[:, s:e].cpu().numpy())
    torch.cuda.synchronize()
    for name in ("k", "v"):
        got = getattr(gc, name)[:, :, :L].cpu().numpy()
        want = getattr(oc, name.upper())[:, :, :L]
        assert got.tobytes() == want.tobytes(), name
    if dtype == kvd.INT8:
        assert gc.k_scale[:, :, :L].cpu().numpy().tobytes() == oc.ks[:, :, :L].tobytes()
    nb = (L + 63) // 64
    assert gc.t["kbounds"][:, :, :nb].cpu().numpy()[..., 0].tobytes() == \
        oc.kmin[:, :, :nb].tobytes()
    assert gc.t["kbounds"][:, :, :nb].cpu().numpy()[..., 1].tobytes() == \
        oc.kmax[:, :, :nb].tobytes()


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("D,G", CASES)
def test_select_and_decode(dtype, D, G):
    B, Hkv, L = 2, 2, 64 * 37 + 13
    k = seeded((B, L, Hkv, D), 100 + D + G, scale=1.5)
    v = seeded((B, L, Hkv, D), 200 + D + G)
    gc, oc = make_pair(dtype, k, v)
    q = seeded((B, Hkv * G, D), 300 + D + G, scale=2.0, dtype=torch.float32)
    ws = kvd.make_workspace(gc, Hkv * G)
    nbmax = gc.max_seq // 64
    sel_idx = torch.full((B, Hkv, nbmax), -1, dtype=torch.int32, device=dev())
    sel_cnt = torch.zeros((B, Hkv), dtype=torch.int32, device=dev())
    k_sel, sink, recent = 7, 4, 100
    kvd.select_blocks(gc, q, k_sel, sink, recent, sel_idx, sel_cnt, ws)
    torch.cuda.synchronize()
    check_selection(sel_idx, sel_cnt, oc, q.cpu().numpy(), k_sel, sink, recent, G)
    out = torch.full((B, Hkv * G, D), float("nan"), device=dev())
    max_sel = kvd.selected_count(L, k_sel, sink, recent)
    kvd.decode_attn(gc, q, scale_for(D), sel_idx, sel_cnt, max_sel, out, ws)
    torch.cuda.synchronize()
    assert gc.device_status() == 0
    _check_outputs(dtype, gc, oc, q, out, G, D, sel_idx, sel_cnt, f"sparse D{D} G{G}")
    again = torch.empty_like(out)
    kvd.decode_attn(gc, q, scale_for(D), sel_idx, sel_cnt, max_sel, again, ws)
    torch.cuda.synchronize()
    assert torch.equal(out, again)
    dense = torch.full_like(out, float("nan"))
    kvd.decode_attn_dense(gc, q, scale_for(D), dense, ws)
    torch.cuda.synchronize()
    _check_outputs(dtype, gc, oc, q, dense, G, D, what=f"dense D{D} G{G}")


@pytest.mark.parametrize("dtype", DTYPES)
def test_edge_cases(dtype):
    D, G, Hkv = 64, 4, 2
    # one token: a single ragged block
    k = seeded((1, 1, Hkv, D), 31)
    v = seeded((1, 1, Hkv, D), 32)
    gc, oc = make_pair(dtype, k, v, max_seq=128)
    q = seeded((1, Hkv * G, D), 33, dtype=torch.float32)
    ws = kvd.make_workspace(gc, Hkv * G)
    out = torch.empty(1, Hkv * G, D, device=dev())
    kvd.decode_attn_dense(gc, q, scale_for(D), out, ws)
    torch.cuda.synchronize()
    _check_outputs(dtype, gc, oc, q, out, G, D, what="one token")
    # every candidate selected; and an empty selection gives zeros
    L = 64 * 9 + 5
    k = seeded((1, L, Hkv, D), 34)
    v = seeded((1, L, Hkv, D), 35)
    gc, oc = make_pair(dtype, k, v)
    ws = kvd.make_workspace(gc, Hkv * G)
    nbmax = gc.max_seq // 64
    sel_idx = torch.zeros((1, Hkv, nbmax), dtype=torch.int32, device=dev())
    sel_cnt = torch.zeros((1, Hkv), dtype=torch.int32, device=dev())
    kvd.select_blocks(gc, q, 100, 0, 0, sel_idx, sel_cnt, ws)
    torch.cuda.synchronize()
    assert sel_cnt.cpu().tolist() == [[10, 10]]
    assert sel_idx[0, :, :10].cpu().tolist() == [list(range(10))] * 2
    kvd.select_blocks(gc, q, 0, 0, 0, sel_idx, sel_cnt, ws)
    out = torch.full((1, Hkv * G, D), float("nan"), device=dev())
    kvd.decode_attn(gc, q, scale_for(D), sel_idx, sel_cnt, 1, out, ws)
    torch.cuda.synchronize()
    assert sel_cnt.cpu().tolist() == [[0, 0]]
    assert torch.count_nonzero(out).item() == 0
    # a bad block id in a caller's list is skipped and reported
    sel_idx[0, :, 0] = 3
    sel_idx[0, :, 1] = 999
    sel_cnt.fill_(2)
    kvd.decode_attn(gc, q, scale_for(D), sel_idx, sel_cnt, 2, out, ws)
    torch.cuda.synchronize()
    assert gc.device_status() == 1
    _check_outputs(dtype, gc, oc, q, out, G, D, sel_idx[:, :, :1].contiguous(),
                   torch.ones_like(sel_cnt), "bad id skipped")


def test_equal_bounds_take_the_lowest_index():
    # identical keys in every block: all bounds tie, so the top K are the
    # lowest candidate indices
    D, G, Hkv, L = 96, 2, 1, 64 * 20
    row = seeded((1, 1, Hkv, D), 41)
    k = row.expand(1, L, Hkv, D).contiguous()
    v = seeded((1, L, Hkv, D), 42)
    gc, oc = make_pair(kvd.INT8, k, v)
    q = seeded((1, Hkv * G, D), 43, dtype=torch.float32)
    ws = kvd.make_workspace(gc, Hkv * G)
    nbmax = gc.max_seq // 64
    sel_idx = torch.zeros((1, Hkv, nbmax), dtype=torch.int32, device=dev())
    sel_cnt = torch.zeros((1, Hkv), dtype=torch.int32, device=dev())
    kvd.select_blocks(gc, q, 5, 64, 64, sel_idx, sel_cnt, ws)
    torch.cuda.synchronize()
    assert sel_idx[0, 0, :int(sel_cnt[0, 0])].cpu().tolist() == [0, 1, 2, 3, 4, 5, 19]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("D,G,dense", [(64, 4, False), (256, 8, False), (112, 2, True)])
def test_decode_steps(dtype, D, G, dense):
    B, Hkv, L = 2, 2, 64 * 12 + 40
    k = seeded((B, L, Hkv, D), 500 + D, scale=1.5)
    v = seeded((B, L, Hkv, D), 600 + D)
    gc, oc = make_pair(dtype, k, v, max_seq=64 * 14)
    ws = kvd.make_workspace(gc, Hkv * G)
    nbmax = gc.max_seq // 64
    sel_idx = torch.zeros((B, Hkv, nbmax), dtype=torch.int32, device=dev())
    sel_cnt = torch.zeros((B, Hkv), dtype=torch.int32, device=dev())
    out = torch.empty((B, Hkv * G, D), device=dev())
    k_sel = -1 if dense else 3
    for step in range(3):
        q = seeded((B, Hkv * G, D), 700 + step, scale=2.0, dtype=torch.float32)
        kn = seeded((B, 1, Hkv, D), 800 + step)
        vn = seeded((B, 1, Hkv, D), 900 + step)
        kvd.decode_step(gc, q, kn, vn, scale_for(D), k_sel, 4, 64, out, ws, sel_idx, sel_cnt)
        oc.append(kn.cpu().numpy(), vn.cpu().numpy())
        torch.cuda.synchronize()
        assert gc.device_status() == 0 and gc.len == oc.len
        if dense:
            _check_outputs(dtype, gc, oc, q, out, G, D, what=f"dense step {step}")
        else:
            check_selection(sel_idx, sel_cnt, oc, q.cpu().numpy(), k_sel, 4, 64, G)
            _check_outputs(dtype, gc, oc, q, out, G, D, sel_idx, sel_cnt, f"step {step}")


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("D,pinned", [(96, "none"), (256, "mixed"), (48, "all")])
def test_host_step_equals_device_step(dtype, D, pinned):
    # the host-buffer step stages (or maps) D-channel rows and equals the
    # device step bit for bit
    B, Hkv, G, L0 = 2, 2, 4, 64 * 9 + 7
    k = seeded((B, L0, Hkv, D), 41 + D)
    v = seeded((B, L0, Hkv, D), 42 + D)
    a, _ = make_pair(dtype, k, v, max_seq=64 * 11)
    b, _ = make_pair(dtype, k, v, max_seq=64 * 11)
    wa = kvd.make_workspace(a, Hkv * G)
    wb = kvd.make_workspace(b, Hkv * G)
    for s in range(3):
        q = seeded((B, Hkv * G, D), 50 + s, dtype=torch.float32)
        kn = seeded((B, 1, Hkv, D), 60 + s)
        vn = seeded((B, 1, Hkv, D), 70 + s)
        out_d = torch.empty(B, Hkv * G, D, device=dev())
        kvd.decode_step(a, q, kn, vn, scale_for(D), 3, 4, 64, out_d, wa)
        pin = {"all": (1, 1, 1, 1), "none": (0, 0, 0, 0), "mixed": (1, 0, 1, 0)}[pinned]
        qh, kh, vh = (t.cpu().pin_memory() if p else t.cpu().clone()
                      for t, p in zip((q, kn, vn), pin[:3]))
        out_h = torch.empty(B, Hkv * G, D)
        out_h = out_h.pin_memory() if pin[3] else out_h
        kvd.decode_step_host(b, qh, kh, vh, scale_for(D), 3, 4, 64, out_h, wb)
        torch.cuda.synchronize()
        assert torch.equal(out_d.cpu(), out_h)
    assert a.len == b.len == L0 + 3
    assert a.device_status() == b.device_status() == 0


@pytest.mark.parametrize("D", [256, 512])
def test_repeated_steps_with_tiles_past_the_end(D):
    # The fast kernel cuts a block into several tiles at these dims; the last
    # block of a sequence ending one token into it leaves tiles past the end,
    # whose stages complete at once.  Many steps over the same cache (the
    # length reset each time, as the bench does) must never run into the
    # kernel's bounded wait, and repeat bit for bit.
    B, Hkv, G, L0 = 1, 8, 4, 64 * 200
    k = seeded((B, L0, Hkv, D), 31 + D)
    v = seeded((B, L0, Hkv, D), 32 + D)
    gc = kvd.KVCache(kvd.F16, B, Hkv, L0 + 64, head_dim=D, device=dev())
    kvd.kv_append(gc, k, v)
    ws = kvd.make_workspace(gc, Hkv * G)
    q = seeded((B, Hkv * G, D), 33 + D, scale=2.0, dtype=torch.float32)
    kn = seeded((B, 1, Hkv, D), 34 + D)
    vn = seeded((B, 1, Hkv, D), 35 + D)
    out = torch.empty((B, Hkv * G, D), device=dev())
    first = None
    for step in range(300):
        gc.len = L0
        kvd.decode_step(gc, q, kn, vn, scale_for(D), 40, 4, 64, out, ws)
        if step == 0:
            torch.cuda.synchronize()
            first = out.clone()
    torch.cuda.synchronize()
    assert gc.device_status() == 0
    assert torch.equal(out, first)
