"""The C ABI library loads and rejects bad arguments on the host (no GPU).

Every call below fails validation, so nothing reaches the CUDA runtime; a
call that passed validation on a machine without a GPU would return
KVD_ERR_CUDA, which these tests would flag.
"""
import ctypes as C
import os
import re

import numpy as np
import pytest

import long_context_decode_kv_gb300 as kvd
from long_context_decode_kv_gb300 import CacheStruct

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvdecode.h")

OK, INVALID, UNSUPPORTED, CAPACITY, CUDA, TIMEOUT, WORKSPACE = range(7)
FAKE = 0x7f0000000000  # aligned, never dereferenced on the host


@pytest.fixture(scope="module", autouse=True)
def _built():
    from long_context_decode_kv_gb300 import build
    build.build()


def _cache(dtype=kvd.INT8, B=1, Hkv=8, D=128, max_seq=4096, blk=64, length=1000, **kw):
    s = CacheStruct(dtype, B, Hkv, D, max_seq, blk, length, 0, FAKE, FAKE + 0x100000,
                    FAKE + 0x200000, FAKE + 0x300000, FAKE + 0x400000, None)
    for k, v in kw.items():
        setattr(s, k, v)
    return s


def test_header_symbols_exported():
    decl = re.findall(r"^KVD_API\s+[\w\s\*]+?\b(kvd_\w+)\s*\(", open(HEADER).read(), re.M)
    assert len(decl) >= 12
    L = C.CDLL(kvd.LIB_PATH)
    for name in decl:
        assert hasattr(L, name), name
    assert set(decl) == set(kvd.EXPORTS)


def test_abi_version_and_status_strings():
    v = int(re.search(r"#define KVD_ABI_VERSION (\d+)", open(HEADER).read()).group(1))
    assert kvd.lib().kvd_abi_version() == v
    for code in range(7):
        assert kvd.status_string(code) and kvd.status_string(code) != "unknown status"
    assert kvd.status_string(99) == "unknown status"


def test_selected_count_matches_oracle_rule():
    import oracle
    rng = np.random.default_rng(5)
    for _ in range(300):
        L = int(rng.integers(1, 5000))
        k = int(rng.integers(0, 100))
        sink = int(rng.integers(0, 300))
        rec = int(rng.integers(0, 300))
        nb = (L + 63) // 64
        sel, _ = oracle.select(L, 64, np.zeros(nb), k, sink, rec)
        assert kvd.selected_count(L, k, sink, rec) == len(sel)
    assert kvd.selected_count(0, 1, 0, 0) == -1
    assert kvd.selected_count(10, -1, 0, 0) == -1
    assert kvd.selected_count(10, 1, 0, 0, block=32) == -1


def _ws(s, n_heads=32):
    return int(kvd.lib().kvd_workspace_bytes(C.byref(s), n_heads))


def test_workspace_bytes():
    s = _cache()
    n = _ws(s)
    assert n > 0 and n % 256 == 0
    assert _ws(_cache(max_seq=8192)) > n           # grows with capacity
    assert _ws(s, 33) == 0                          # 33 % 8 != 0
    assert _ws(_cache(D=72)) == 0                   # D not a multiple of 16
    assert _ws(_cache(dtype=7)) == 0


def _select(s, n_heads=32, k_sel=4, sink=4, recent=64, ws_bytes=None, q=FAKE, ws=FAKE):
    ws_bytes = _ws(_cache()) if ws_bytes is None else ws_bytes
    return kvd.lib().kvd_select_blocks(C.byref(s), q, n_heads, k_sel, sink, recent, FAKE, FAKE,
                                       ws, ws_bytes, None)


def test_select_validation():
    assert _select(_cache(D=72)) == UNSUPPORTED              # not a multiple of 16
    assert _select(_cache(D=1040)) == UNSUPPORTED            # above 1024
    assert _select(_cache(D=0)) == UNSUPPORTED
    assert _select(_cache(dtype=kvd.Q8_0, D=64)) == UNSUPPORTED  # group types: D = 128
    assert _select(_cache(D=64, moments=FAKE)) == UNSUPPORTED    # block means: D = 128
    assert _select(_cache(D=64, seq_lens=FAKE)) == UNSUPPORTED   # per-sequence: D = 128
    assert _select(_cache(blk=32)) == UNSUPPORTED
    assert _select(_cache(), n_heads=12) == INVALID
    assert _select(_cache(), n_heads=24) == UNSUPPORTED      # group of 3
    assert _select(_cache(length=0)) == INVALID
    assert _select(_cache(), k_sel=-1) == INVALID
    assert _select(_cache(), sink=-1) == INVALID
    assert _select(_cache(), recent=-1) == INVALID
    assert _select(_cache(), q=FAKE + 4) == INVALID          # misaligned q
    assert _select(_cache(), q=None) == INVALID
    assert _select(_cache(), ws_bytes=16) == WORKSPACE
    assert _select(_cache(), ws=FAKE + 8) == WORKSPACE
    assert _select(_cache(), ws=None) == WORKSPACE
    assert _select(_cache(k=FAKE + 2)) == INVALID
    assert _select(_cache(kbounds=None)) == INVALID
    assert _select(_cache(k_scale=None)) == INVALID
    for dt in (kvd.Q8_0, kvd.Q4_0):                         # group scales required
        assert _select(_cache(dtype=dt, k_scale=None)) == INVALID
        assert _select(_cache(dtype=dt, v_scale=None)) == INVALID
    assert _select(_cache(max_seq=100)) == INVALID           # not a multiple of 64
    assert _select(_cache(length=5000)) == INVALID           # len > max_seq
    assert _select(_cache(reserved=1)) == INVALID
    big = _cache(max_seq=64 * 49153, length=64 * 49153)
    assert _select(big, ws_bytes=_ws(big)) == UNSUPPORTED     # too many blocks to select


def test_decode_validation():
    L = kvd.lib()
    s = _cache()
    n = _ws(s)
    assert L.kvd_decode_attn(C.byref(_cache(length=0)), FAKE, 32, 0.1, FAKE, FAKE, 10, FAKE,
                             FAKE, n, None) == INVALID
    assert L.kvd_decode_attn(C.byref(s), FAKE, 32, 0.1, None, FAKE, 10, FAKE, FAKE, n,
                             None) == INVALID
    assert L.kvd_decode_attn(C.byref(s), FAKE, 32, 0.1, FAKE, FAKE, -1, FAKE, FAKE, n,
                             None) == INVALID
    assert L.kvd_decode_attn(C.byref(s), FAKE, 32, 0.1, FAKE, FAKE, 10, FAKE + 4, FAKE, n,
                             None) == INVALID
    assert L.kvd_decode_attn(C.byref(s), FAKE, 32, 0.1, FAKE, FAKE, 10, FAKE, FAKE, n - 256,
                             None) == WORKSPACE
    assert L.kvd_decode_attn_dense(C.byref(s), FAKE, 30, 0.1, FAKE, FAKE, n, None) == INVALID
    assert L.kvd_decode_attn_dense(C.byref(_cache(head_dim=264)), FAKE, 32, 0.1, FAKE, FAKE, n,
                                   None) == UNSUPPORTED
    assert L.kvd_decode_attn_dense(C.byref(s), FAKE, 32, 0.1, FAKE, None, n, None) == WORKSPACE


def test_decode_tail_validation():
    L = kvd.lib()
    s = _cache(moments=FAKE + 0x500000)
    n = _ws(s)
    tail = L.kvd_decode_attn_tail
    assert tail(C.byref(_cache()), FAKE, 32, 0.1, FAKE, FAKE, 10, FAKE, FAKE, n,
                None) == INVALID                                   # no moments kept
    assert tail(C.byref(_cache(moments=FAKE + 8)), FAKE, 32, 0.1, FAKE, FAKE, 10, FAKE, FAKE,
                n, None) == INVALID                                # misaligned moments
    assert tail(C.byref(s), FAKE, 32, 0.1, None, FAKE, 10, FAKE, FAKE, n, None) == INVALID
    assert tail(C.byref(s), FAKE, 32, 0.1, FAKE, None, 10, FAKE, FAKE, n, None) == INVALID
    assert tail(C.byref(s), FAKE, 32, 0.1, FAKE, FAKE, -1, FAKE, FAKE, n, None) == INVALID
    assert tail(C.byref(_cache(moments=FAKE + 0x500000, length=0)), FAKE, 32, 0.1, FAKE, FAKE,
                10, FAKE, FAKE, n, None) == INVALID
    assert tail(C.byref(s), FAKE, 32, 0.1, FAKE, FAKE, 10, FAKE, FAKE, n - 256,
                None) == WORKSPACE
    # per-head selection and decode validate like the shared calls
    ph = L.kvd_select_blocks_per_head
    assert ph(C.byref(s), FAKE, 12, 4, 4, 64, FAKE, FAKE, FAKE, n, None) == INVALID
    assert ph(C.byref(s), FAKE, 32, -1, 4, 64, FAKE, FAKE, FAKE, n, None) == INVALID
    assert ph(C.byref(s), FAKE, 32, 4, 4, 64, None, FAKE, FAKE, n, None) == INVALID
    assert ph(C.byref(s), FAKE, 32, 4, 4, 64, FAKE, FAKE, FAKE, 16, None) == WORKSPACE
    pd = L.kvd_decode_attn_per_head
    assert pd(C.byref(s), FAKE, 32, 0.1, FAKE, None, 10, FAKE, FAKE, n, None) == INVALID
    assert pd(C.byref(s), FAKE, 32, 0.1, FAKE, FAKE, -1, FAKE, FAKE, n, None) == INVALID
    assert pd(C.byref(s), FAKE, 32, 0.1, FAKE, FAKE, 10, FAKE, None, n, None) == WORKSPACE
    # per-sequence lengths: aligned, and not taken by the whole-step calls
    assert _select(_cache(seq_lens=FAKE + 2)) == INVALID
    assert L.kvd_decode_step(C.byref(_cache(seq_lens=FAKE + 2)), FAKE, FAKE, FAKE, 32, 0.1, 4,
                             4, 64, None, None, FAKE, FAKE, n, None) == INVALID
    assert L.kvd_debug_scores(C.byref(_cache(seq_lens=FAKE)), FAKE, 32, FAKE,
                              None) == UNSUPPORTED
    # a cache that keeps moments is otherwise an ordinary cache
    assert _select(_cache(moments=FAKE + 8)) == INVALID


def test_general_head_dims():
    L = kvd.lib()
    for D in (16, 64, 80, 96, 256, 1024):
        for dt in (kvd.F16, kvd.INT8):
            s = _cache(dtype=dt, D=D)
            need = L.kvd_workspace_bytes(C.byref(s), 32)
            assert need > 0 and need % 256 == 0, (D, dt)
            # validation runs first and still applies
            assert _select(s, n_heads=24, ws_bytes=need) == UNSUPPORTED
            assert _select(s, k_sel=-1, ws_bytes=need) == INVALID
            assert _select(s, ws_bytes=need - 256) == WORKSPACE
    big = L.kvd_workspace_bytes(C.byref(_cache(D=1024)), 32)
    assert big > L.kvd_workspace_bytes(C.byref(_cache(D=64)), 32)
    assert L.kvd_workspace_bytes(C.byref(_cache(D=72)), 32) == 0
    s = _cache(D=64)
    n = L.kvd_workspace_bytes(C.byref(s), 32)
    # the calls only the D = 128 kernels serve
    assert L.kvd_select_blocks_per_head(C.byref(s), FAKE, 32, 4, 4, 64, FAKE, FAKE, FAKE, n,
                                        None) == UNSUPPORTED
    assert L.kvd_decode_attn_per_head(C.byref(s), FAKE, 32, 0.1, FAKE, FAKE, 10, FAKE, FAKE, n,
                                      None) == UNSUPPORTED
    assert L.kvd_debug_scores(C.byref(s), FAKE, 32, FAKE, None) == UNSUPPORTED
    assert L.kvd_debug_qk_int8(C.byref(s), FAKE, 32, FAKE, FAKE, FAKE, None) == UNSUPPORTED
    # sparse-V with eps > 0 is a tuned-kernel mode (refused before any launch)
    assert L.kvd_decode_attn_sv(C.byref(s), FAKE, 32, 0.1, FAKE, FAKE, 10, 0.5, FAKE, FAKE, n,
                                None) == UNSUPPORTED


def test_wait_timeout_validation():
    L = kvd.lib()
    assert L.kvd_debug_wait_timeout(None, 1000, None) == INVALID
    assert L.kvd_debug_wait_timeout(FAKE + 2, 1000, None) == INVALID
    assert L.kvd_debug_wait_timeout(FAKE, 0, None) == INVALID
    assert L.kvd_debug_wait_timeout(FAKE, 1000001, None) == INVALID
    # stage marks exist only in a library built with KVD_MARKS=1
    assert L.kvd_debug_stage_marks(FAKE, 3 * 4096 * 16 * 8) == UNSUPPORTED


def test_append_validation():
    L = kvd.lib()
    s = _cache(length=4090)
    assert L.kvd_kv_append(C.byref(s), FAKE, FAKE, 7, None) == CAPACITY
    assert s.len == 4090
    assert L.kvd_kv_append(C.byref(s), FAKE, FAKE, -1, None) == INVALID
    assert L.kvd_kv_append(C.byref(s), FAKE, FAKE, 0, None) == OK      # no-op, no launch
    assert s.len == 4090
    assert L.kvd_kv_append(C.byref(s), FAKE + 2, FAKE, 1, None) == INVALID
    assert L.kvd_kv_append(C.byref(s), None, FAKE, 1, None) == INVALID
    assert L.kvd_kv_append(C.byref(_cache(dtype=7)), FAKE, FAKE, 1, None) == INVALID
    s = _cache(length=4090)
    assert L.kvd_kv_append_f32(C.byref(s), FAKE, FAKE, 7, None) == CAPACITY
    assert L.kvd_kv_append_f32(C.byref(s), FAKE + 8, FAKE, 1, None) == INVALID
    assert L.kvd_kv_append_f32(C.byref(s), FAKE, None, 1, None) == INVALID
    assert L.kvd_kv_append_f32(C.byref(s), FAKE, FAKE, 0, None) == OK
    assert s.len == 4090
    assert L.kvd_kv_append(C.byref(None if False else _cache(n_kv_heads=0)), FAKE, FAKE, 1,
                           None) == INVALID


def test_step_validation():
    L = kvd.lib()
    s = _cache(length=4096)
    n = _ws(s)
    assert L.kvd_decode_step(C.byref(s), FAKE, FAKE, FAKE, 32, 0.1, 4, 4, 64, None, None, FAKE,
                             FAKE, n, None) == CAPACITY
    s = _cache()
    assert L.kvd_decode_step(C.byref(s), FAKE, FAKE, FAKE, 32, 0.1, 4, -4, 64, None, None, FAKE,
                             FAKE, n, None) == INVALID
    assert L.kvd_decode_step(C.byref(s), FAKE, FAKE, FAKE, 32, 0.1, 4, 4, 64, None, None, FAKE,
                             FAKE, 64, None) == WORKSPACE
    assert s.len == 1000
    assert L.kvd_decode_step_host(C.byref(s), None, FAKE, FAKE, 32, 0.1, 4, 4, 64, None, None,
                                  FAKE, FAKE, n, None) == INVALID


def test_debug_validation():
    L = kvd.lib()
    assert L.kvd_debug_qk_int8(C.byref(_cache(dtype=kvd.F16)), FAKE, 32, FAKE, FAKE, FAKE,
                               None) == INVALID
    assert L.kvd_debug_scores(C.byref(_cache(length=0)), FAKE, 32, FAKE, None) == INVALID
    assert L.kvd_debug_scores(C.byref(_cache()), FAKE, 32, None, None) == INVALID


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import importlib
    mod = importlib.reload(kvd)
    monkeypatch.setattr(mod, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(mod, "_lib", None)
    with pytest.raises(ImportError):
        mod.lib()
    importlib.reload(kvd)
