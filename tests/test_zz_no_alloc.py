"""kvd_decode_attn_static: the decode without a caller workspace.

Its scratch is a fixed array inside the library, shared by every call on the
device, so the GPU test makes two calls in a row (different caches, queries and
split grids) and checks each against kvd_decode_attn on the same inputs with
the decode tests' bar: relative L2 per (sequence, query head) within 2e-3 (f16)
/ 8e-3 (int8) and within 1e-4.  The file is named to be collected last, and the
test holds whether it runs alone in a fresh process or after the others.
"""
import ctypes as C

import pytest
import torch

import long_context_decode_kv_gb300 as kvd

OK, INVALID, UNSUPPORTED = 0, 1, 2
FAKE = 0x7f0000000000  # aligned, never dereferenced on the host


def _fake_cache(**kw):
    s = kvd.CacheStruct(kvd.INT8, 1, 8, 128, 4096, 64, 1000, 0, FAKE, FAKE + 0x100000,
                    FAKE + 0x200000, FAKE + 0x300000, FAKE + 0x400000, None)
    for k, v in kw.items():
        setattr(s, k, v)
    return s


def test_static_validation_on_host():
    from long_context_decode_kv_gb300 import build
    build.build()
    L = kvd.lib()

    def call(s, q=FAKE, n_heads=32, idx=FAKE, cnt=FAKE, max_sel=10, out=FAKE):
        return L.kvd_decode_attn_static(C.byref(s), q, n_heads, 0.1, idx, cnt, max_sel, out,
                                        None)

    assert call(_fake_cache(len=0)) == INVALID
    assert call(_fake_cache(head_dim=64)) == UNSUPPORTED
    assert call(_fake_cache(), n_heads=12) == INVALID
    assert call(_fake_cache(), n_heads=24) == UNSUPPORTED
    assert call(_fake_cache(), idx=None) == INVALID
    assert call(_fake_cache(), cnt=FAKE + 2) == INVALID
    assert call(_fake_cache(), max_sel=-1) == INVALID
    assert call(_fake_cache(), q=FAKE + 4) == INVALID
    assert call(_fake_cache(), out=None) == INVALID
    assert call(_fake_cache(k_scale=None)) == INVALID
    assert call(_fake_cache(reserved=1)) == INVALID


def _case(dtype, B, Hkv, G, L, k_sel, sink, recent, seed):
    """A filled cache, a query and a selection made by kvd_select_blocks."""
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    k = (torch.randn(B, L, Hkv, 128, generator=g, device=dev) * 1.5).half()
    v = torch.randn(B, L, Hkv, 128, generator=g, device=dev).half()
    q = torch.randn(B, Hkv * G, 128, generator=g, device=dev)
    cache = kvd.KVCache(dtype, B, Hkv, (L + 64 + 63) // 64 * 64, device=dev)
    kvd.kv_append(cache, k, v)
    ws = kvd.make_workspace(cache, Hkv * G)
    nbmax = cache.max_seq // 64
    sel_idx = torch.zeros(B, Hkv, nbmax, dtype=torch.int32, device=dev)
    sel_cnt = torch.zeros(B, Hkv, dtype=torch.int32, device=dev)
    kvd.select_blocks(cache, q, k_sel, sink, recent, sel_idx, sel_cnt, ws)
    max_sel = kvd.selected_count(L, k_sel, sink, recent)
    return cache, q, ws, sel_idx, sel_cnt, max_sel


def _rel_l2(a, b):
    a = a.double().reshape(-1, 128)
    b = b.double().reshape(-1, 128)
    den = b.norm(dim=1).clamp_min(1e-300)
    return ((a - b).norm(dim=1) / den).max().item()


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", [kvd.F16, kvd.INT8])
def test_static_matches_workspace_decode_two_calls(dtype):
    tol = {kvd.F16: 2e-3, kvd.INT8: 8e-3}[dtype]
    scale = 128 ** -0.5
    cases = [
        _case(dtype, 1, 8, 8, 40000, 120, 64, 1024, 901),   # many splits, 2 subgroups
        _case(dtype, 3, 2, 4, 5000, 16, 4, 256, 902),       # other grid, other layout
    ]
    refs, outs = [], []
    for cache, q, ws, sel_idx, sel_cnt, max_sel in cases:
        ref = torch.full_like(q, float("nan"))
        kvd.decode_attn(cache, q, scale, sel_idx, sel_cnt, max_sel, ref, ws)
        refs.append(ref)
        outs.append(torch.full_like(q, float("nan")))
    torch.cuda.synchronize()

    # two calls in a row on the shared array, each checked against the workspace path
    for _ in range(2):
        allocated = torch.cuda.memory_allocated()
        for (cache, q, _ws, sel_idx, sel_cnt, max_sel), out in zip(cases, outs):
            out.fill_(float("nan"))
            kvd.decode_attn_static(cache, q, scale, sel_idx, sel_cnt, max_sel, out)
        torch.cuda.synchronize()
        assert torch.cuda.memory_allocated() == allocated
        for i, (out, ref) in enumerate(zip(outs, refs)):
            assert torch.isfinite(out).all(), f"case {i}"
            e = _rel_l2(out, ref)
            assert e <= tol and e <= 1e-4, f"case {i}: rel L2 {e:.3e}"


@pytest.mark.gpu
def test_static_extreme_shapes_two_calls():
    # the shapes that size the array: the most problems the decode accepts
    # (batch * KV heads * 16 <= 65535, here 4095 problems of 16 query heads:
    # the most arrival counters), and a grid just under one wave of two CTAs
    # per SM with two splits each (the most split partials, ~0.65 MiB on 152 SMs)
    scale = 128 ** -0.5
    cases = [
        (kvd.F16, _case(kvd.F16, 4095, 1, 16, 100, 1, 0, 0, 903)),
        (kvd.INT8, _case(kvd.INT8, 1, 38, 16, 2048, 24, 4, 64, 904)),
    ]
    refs = []
    for _, (cache, q, ws, sel_idx, sel_cnt, max_sel) in cases:
        ref = torch.full_like(q, float("nan"))
        kvd.decode_attn(cache, q, scale, sel_idx, sel_cnt, max_sel, ref, ws)
        refs.append(ref)
    torch.cuda.synchronize()
    for _ in range(2):
        for (dtype, (cache, q, _ws, sel_idx, sel_cnt, max_sel)), ref in zip(cases, refs):
            out = torch.full_like(q, float("nan"))
            kvd.decode_attn_static(cache, q, scale, sel_idx, sel_cnt, max_sel, out)
            torch.cuda.synchronize()
            assert torch.isfinite(out).all()
            e = _rel_l2(out, ref)
            assert e <= {kvd.F16: 2e-3, kvd.INT8: 8e-3}[dtype] and e <= 1e-4, e
