"""fp64 CPU oracle for Quest-style sparse decode attention (ctypes over ``oracle.c``).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  It shares no
code with the CUDA library; both sides only read the same seeded inputs.

Every routine restates a passage of the pages (cited in ``oracle.c``):
the Quest block bound and top-K selection with sink/recent blocks from the
"Quest-style block-selector for long-context decode" page, and the absmax
int8 cache and decode math from the "cpu-attn" card.  Arrays are numpy:
f16 data travel as ``np.float16`` (bit patterns are passed through
untouched), scales as ``np.float32``, results come back as ``np.float64``.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import build as _build

F16 = 0
INT8 = 1
Q8_0 = 2
Q4_0 = 3
QGROUP = 32

_lib = None


def lib():
    global _lib
    if _lib is None:
        # ORACLE_LIB lets the mutation tests load a deliberately broken copy
        path = os.environ.get("ORACLE_LIB") or _build.build()
        L = C.CDLL(path)
        p = C.c_void_p
        i = C.c_int
        d = C.c_double
        L.orc_half_to_double.argtypes = [C.c_uint16]
        L.orc_half_to_double.restype = d
        L.orc_quantize_row.argtypes = [p, i, p, p]
        L.orc_append.argtypes = [p, p, p, i]
        L.orc_append.restype = i
        L.orc_block_scores.argtypes = [i, i, i, p, p, p, p, p, p]
        L.orc_forced_range.argtypes = [i, i, i, i, p, p]
        L.orc_select.argtypes = [i, i, p, i, i, i, p, p]
        L.orc_select.restype = i
        L.orc_attend_f16.argtypes = [i, i, i, p, d, p, p, p, i, p]
        L.orc_qk_int8.argtypes = [i, C.c_long, p, p, p]
        L.orc_attend_int8.argtypes = [i, i, i, p, C.c_float, d, p, p, p, p, p, i, p]
        L.orc_attend_dequant.argtypes = [i, i, i, p, p, C.c_float, d, p, p, p, p, p, i, p]
        L.orc_sparse_v_keep.argtypes = [C.c_long, p, p, d, p]
        L.orc_double_to_half.argtypes = [d]
        L.orc_double_to_half.restype = C.c_uint16
        L.orc_quantize_group32.argtypes = [p, i, p, p]
        L.orc_attend_q8_0.argtypes = [i, i, i, p, C.c_float, d, p, p, p, p, p, i, d, p, p]
        L.orc_quantize_q4_0.argtypes = [p, i, p, p]
        L.orc_attend_q4_0.argtypes = [i, i, i, p, C.c_float, d, p, p, p, p, p, i, d, p, p]
        L.orc_attend_f16_sv.argtypes = [i, i, i, p, d, p, p, p, i, d, p, p]
        L.orc_attend_int8_sv.argtypes = [i, i, i, p, C.c_float, d, p, p, p, p, p, i, d, p, p]
        L.orc_block_moments.argtypes = [i, i, i, p, p]
        L.orc_append_f32.argtypes = [p, p, p, i]
        L.orc_append_f32.restype = i
        L.orc_double_to_half_dir.argtypes = [d, i]
        L.orc_double_to_half_dir.restype = C.c_uint16
        L.orc_attend_tail.argtypes = [i, i, i, p, p, d, p, p, p, i, p, p, p]
        L.orc_decode.argtypes = [p, i, p, d, i, i, i, i, p, p, p, i]
        L.orc_decode.restype = i
        L.orc_num_threads_available.restype = i
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


class _OrcCache(C.Structure):
    _fields_ = [("dtype", C.c_int), ("B", C.c_int), ("Hkv", C.c_int), ("D", C.c_int),
                ("max_seq", C.c_int), ("blk", C.c_int), ("len", C.c_int),
                ("K", C.c_void_p), ("V", C.c_void_p), ("ks", C.c_void_p), ("vs", C.c_void_p),
                ("kmin", C.c_void_p), ("kmax", C.c_void_p), ("kd", C.c_void_p),
                ("vd", C.c_void_p)]


def half_to_double(h) -> float:
    """binary16 bit pattern (int) -> exact float."""
    return lib().orc_half_to_double(int(h) & 0xFFFF)


def quantize_row(x):
    """Absmax int8 codes and f32 scale of one f32 row (cpu-attn, Method)."""
    x = _c(x, np.float32).ravel()
    code = np.zeros(x.size, np.int8)
    scale = np.zeros(1, np.float32)
    lib().orc_quantize_row(_ptr(x), x.size, _ptr(code), _ptr(scale))
    return code, np.float32(scale[0])


class OracleCache:
    """Head-major cache held in numpy arrays, filled by the oracle's own append.

    K, V: [B, Hkv, max_seq, D] (float16, or int8 codes); ks, vs: [B, Hkv,
    max_seq] float32 (int8 only); kd, vd: [B, Hkv, max_seq, D // 32] float16
    group scales (q8_0 and q4_0; q4_0 rows are [.., D // 2] bytes of two codes);
    kmin, kmax: [B, Hkv, max_seq // blk, D] float16.
    """

    def __init__(self, dtype: int, B: int, Hkv: int, D: int, max_seq: int, blk: int = 64):
        assert max_seq % blk == 0
        self.dtype, self.B, self.Hkv, self.D = dtype, B, Hkv, D
        self.max_seq, self.blk, self.len = max_seq, blk, 0
        kvt = np.float16 if dtype == F16 else (np.uint8 if dtype == Q4_0 else np.int8)
        width = D // 2 if dtype == Q4_0 else D
        self.K = np.zeros((B, Hkv, max_seq, width), kvt)
        self.V = np.zeros((B, Hkv, max_seq, width), kvt)
        self.ks = np.zeros((B, Hkv, max_seq), np.float32) if dtype == INT8 else None
        self.vs = np.zeros((B, Hkv, max_seq), np.float32) if dtype == INT8 else None
        q8 = dtype in (Q8_0, Q4_0)
        self.kd = np.zeros((B, Hkv, max_seq, D // QGROUP), np.float16) if q8 else None
        self.vd = np.zeros((B, Hkv, max_seq, D // QGROUP), np.float16) if q8 else None
        nb = max_seq // blk
        self.kmin = np.zeros((B, Hkv, nb, D), np.float16)
        self.kmax = np.zeros((B, Hkv, nb, D), np.float16)

    def _struct(self):
        s = _OrcCache(self.dtype, self.B, self.Hkv, self.D, self.max_seq, self.blk, self.len,
                      _ptr(self.K), _ptr(self.V), _ptr(self.ks), _ptr(self.vs),
                      _ptr(self.kmin), _ptr(self.kmax), _ptr(self.kd), _ptr(self.vd))
        return s

    def append(self, k_new, v_new):
        """k_new, v_new: [B, n_new, Hkv, D] float16."""
        k_new = _c(k_new, np.float16)
        v_new = _c(v_new, np.float16)
        n_new = k_new.shape[1]
        assert k_new.shape == (self.B, n_new, self.Hkv, self.D) == v_new.shape
        s = self._struct()
        rc = lib().orc_append(C.byref(s), _ptr(k_new), _ptr(v_new), n_new)
        if rc != 0:
            raise ValueError("append passes max_seq")
        self.len = s.len

    def append_f32(self, k_new, v_new):
        """k_new, v_new: [B, n_new, Hkv, D] float32 (reading R11)."""
        k_new = _c(k_new, np.float32)
        v_new = _c(v_new, np.float32)
        n_new = k_new.shape[1]
        assert k_new.shape == (self.B, n_new, self.Hkv, self.D) == v_new.shape
        s = self._struct()
        rc = lib().orc_append_f32(C.byref(s), _ptr(k_new), _ptr(v_new), n_new)
        if rc != 0:
            raise ValueError("append passes max_seq")
        self.len = s.len

    def rows(self, b: int, h: int):
        """The stored K and V rows [len, D] of (sequence b, KV head h) in binary64."""
        L = self.len
        sk = self.ks if self.dtype == INT8 else self.kd
        sv = self.vs if self.dtype == INT8 else self.vd
        return (dequant_rows(self.dtype, self.K[b, h, :L], None if sk is None else sk[b, h, :L]),
                dequant_rows(self.dtype, self.V[b, h, :L], None if sv is None else sv[b, h, :L]))

    def moments(self, b: int, h: int):
        """Block means (mK, mV), float16 [ceil(len / blk), D], of (b, h)'s stored rows."""
        K, V = self.rows(b, h)
        return block_moments(K, self.blk), block_moments(V, self.blk)

    def attend_tail(self, b: int, h: int, q, scale: float, sel):
        """One query head over KV head h: the listed blocks exactly, the rest by
        their moment tail.  The exact logits take the query as the cache type's
        decode does (int8 codes for the quantized types); the tail takes it raw."""
        K, V = self.rows(b, h)
        mK, mV = self.moments(b, h)
        q = _c(q, np.float32)
        if self.dtype == F16:
            q_exact = q.astype(np.float64)
        else:
            qc, qs = quantize_row(q)
            q_exact = qc.astype(np.float64) * float(qs)
        return attend_tail(q_exact, q.astype(np.float64), K, V, self.len, self.blk, scale, sel,
                           mK, mV)

    def decode(self, q, scale: float, k_sel: int = 0, sink_tokens: int = 0,
               recent_tokens: int = 0, dense: bool = False, n_threads: int = 1):
        """One decode step: returns (out [B,H,D] f64, sel_idx, sel_cnt)."""
        q = _c(q, np.float32)
        B, H, D = q.shape
        assert B == self.B and D == self.D
        out = np.zeros((B, H, D), np.float64)
        nbmax = self.max_seq // self.blk
        sel_idx = np.full((B, self.Hkv, nbmax), -1, np.int32)
        sel_cnt = np.zeros((B, self.Hkv), np.int32)
        s = self._struct()
        rc = lib().orc_decode(C.byref(s), H, _ptr(q), float(scale), int(k_sel),
                              int(sink_tokens), int(recent_tokens), int(bool(dense)),
                              _ptr(sel_idx), _ptr(sel_cnt), _ptr(out), int(n_threads))
        if rc != 0:
            raise ValueError("bad decode arguments")
        return out, sel_idx, sel_cnt


def block_scores(q, kmin, kmax):
    """Quest bounds of one KV head: (ub [NB], ub_heads [G, NB], mag [NB])."""
    q = _c(q, np.float32)
    if q.ndim == 1:
        q = q[None]
    G, D = q.shape
    kmin = _c(kmin, np.float16)
    kmax = _c(kmax, np.float16)
    NB = kmin.shape[0]
    ub = np.zeros(NB, np.float64)
    ubh = np.zeros((G, NB), np.float64)
    mag = np.zeros(NB, np.float64)
    lib().orc_block_scores(G, D, NB, _ptr(q), _ptr(kmin), _ptr(kmax), _ptr(ubh), _ptr(ub),
                           _ptr(mag))
    return ub, ubh, mag


def forced_range(L, blk, sink_tokens, recent_tokens):
    se = C.c_int()
    rb = C.c_int()
    lib().orc_forced_range(L, blk, sink_tokens, recent_tokens, C.byref(se), C.byref(rb))
    return se.value, rb.value


def select(L, blk, ub, k_sel, sink_tokens, recent_tokens):
    """Selected block ids (ascending) and the bound of the K-th top-K pick."""
    ub = _c(ub, np.float64)
    NB = (L + blk - 1) // blk
    assert ub.size >= NB
    sel = np.zeros(max(NB, 1), np.int32)
    kth = C.c_double()
    n = lib().orc_select(L, blk, _ptr(ub), int(k_sel), int(sink_tokens), int(recent_tokens),
                         _ptr(sel), C.byref(kth))
    return sel[:n].copy(), kth.value


def _sel_args(sel):
    if sel is None:
        return None, -1
    sel = _c(sel, np.int32)
    return sel, sel.size


def attend_f16(q, K, V, L, blk, scale, sel=None):
    q = _c(q, np.float32)
    K = _c(K, np.float16)
    V = _c(V, np.float16)
    D = q.size
    s, n = _sel_args(sel)
    out = np.zeros(D, np.float64)
    lib().orc_attend_f16(D, L, blk, _ptr(q), float(scale), _ptr(K), _ptr(V), _ptr(s), n,
                         _ptr(out))
    return out


def qk_int8(q_code, K):
    q_code = _c(q_code, np.int8)
    K = _c(K, np.int8)
    n, D = K.shape
    dots = np.zeros(n, np.int64)
    lib().orc_qk_int8(D, n, _ptr(q_code), _ptr(K), _ptr(dots))
    return dots


def attend_int8(q_code, q_scale, K, V, ks, vs, L, blk, scale, sel=None):
    q_code = _c(q_code, np.int8)
    K = _c(K, np.int8)
    V = _c(V, np.int8)
    ks = _c(ks, np.float32)
    vs = _c(vs, np.float32)
    D = q_code.size
    s, n = _sel_args(sel)
    out = np.zeros(D, np.float64)
    lib().orc_attend_int8(D, L, blk, _ptr(q_code), float(q_scale), float(scale), _ptr(K),
                          _ptr(V), _ptr(ks), _ptr(vs), _ptr(s), n, _ptr(out))
    return out


def attend_dequant(q, K, V, ks, vs, L, blk, scale, sel=None, q_code=None, q_scale=0.0):
    q = _c(q, np.float32)
    K = _c(K, np.int8)
    V = _c(V, np.int8)
    ks = _c(ks, np.float32)
    vs = _c(vs, np.float32)
    qc = None if q_code is None else _c(q_code, np.int8)
    D = q.size
    s, n = _sel_args(sel)
    out = np.zeros(D, np.float64)
    lib().orc_attend_dequant(D, L, blk, _ptr(q), _ptr(qc), float(q_scale), float(scale),
                             _ptr(K), _ptr(V), _ptr(ks), _ptr(vs), _ptr(s), n, _ptr(out))
    return out


def double_to_half(x) -> np.float16:
    """Nearest binary16 (ties to even), from the oracle's own rounding."""
    return np.array([lib().orc_double_to_half(float(x))], np.uint16).view(np.float16)[0]


def double_to_half_dir(x, direction: int) -> np.float16:
    """The binary16 nearest x toward -inf (direction < 0) or +inf (> 0)."""
    return np.array([lib().orc_double_to_half_dir(float(x), int(direction))],
                    np.uint16).view(np.float16)[0]


def quantize_group32(x):
    """q8_0 codes of a row (length a multiple of 32) and its float16 group scales."""
    x = _c(x, np.float32)
    code = np.zeros(x.size, np.int8)
    d = np.zeros(x.size // QGROUP, np.uint16)
    lib().orc_quantize_group32(_ptr(x), x.size, _ptr(code), _ptr(d))
    return code, d.view(np.float16)


def quantize_q4_0(x):
    """q4_0 packed codes ([n // 2] uint8) of a row and its float16 group scales."""
    x = _c(x, np.float32)
    packed = np.zeros(x.size // 2, np.uint8)
    d = np.zeros(x.size // QGROUP, np.uint16)
    lib().orc_quantize_q4_0(_ptr(x), x.size, _ptr(packed), _ptr(d))
    return packed, d.view(np.float16)


def attend_q4_0(q_code, q_scale, K, V, kd, vd, L, blk, scale, sel=None, eps=0.0):
    """q4_0 attention of one head (sparse-V at eps): (out [D], dropped mass share)."""
    q_code = _c(q_code, np.int8)
    K = _c(K, np.uint8)
    V = _c(V, np.uint8)
    kd = _c(kd, np.float16)
    vd = _c(vd, np.float16)
    D = q_code.size
    s, n = _sel_args(sel)
    out = np.zeros(D, np.float64)
    dropped = C.c_double()
    lib().orc_attend_q4_0(D, L, blk, _ptr(q_code), float(q_scale), float(scale), _ptr(K),
                          _ptr(V), _ptr(kd), _ptr(vd), _ptr(s), n, float(eps), _ptr(out),
                          C.byref(dropped))
    return out, dropped.value


def attend_q8_0(q_code, q_scale, K, V, kd, vd, L, blk, scale, sel=None, eps=0.0):
    """q8_0 attention of one head (sparse-V at eps): (out [D], dropped mass share)."""
    q_code = _c(q_code, np.int8)
    K = _c(K, np.int8)
    V = _c(V, np.int8)
    kd = _c(kd, np.float16)
    vd = _c(vd, np.float16)
    D = q_code.size
    s, n = _sel_args(sel)
    out = np.zeros(D, np.float64)
    dropped = C.c_double()
    lib().orc_attend_q8_0(D, L, blk, _ptr(q_code), float(q_scale), float(scale), _ptr(K),
                          _ptr(V), _ptr(kd), _ptr(vd), _ptr(s), n, float(eps), _ptr(out),
                          C.byref(dropped))
    return out, dropped.value


def sparse_v_keep(tok, lg, eps):
    """Sparse-V keep mask (eps mode) of attended positions tok with logits lg."""
    tok = _c(tok, np.int64)
    lg = _c(lg, np.float64)
    keep = np.zeros(max(tok.size, 1), np.int32)
    lib().orc_sparse_v_keep(tok.size, _ptr(tok), _ptr(lg), float(eps), _ptr(keep))
    return keep[:tok.size].astype(bool)


def attend_f16_sv(q, K, V, L, blk, scale, eps, sel=None):
    """attend_f16 with sparse-V (eps mode): (out [D], dropped mass share)."""
    q = _c(q, np.float32)
    K = _c(K, np.float16)
    V = _c(V, np.float16)
    D = q.size
    s, n = _sel_args(sel)
    out = np.zeros(D, np.float64)
    dropped = C.c_double()
    lib().orc_attend_f16_sv(D, L, blk, _ptr(q), float(scale), _ptr(K), _ptr(V), _ptr(s), n,
                            float(eps), _ptr(out), C.byref(dropped))
    return out, dropped.value


def attend_int8_sv(q_code, q_scale, K, V, ks, vs, L, blk, scale, eps, sel=None):
    """attend_int8 with sparse-V (eps mode): (out [D], dropped mass share)."""
    q_code = _c(q_code, np.int8)
    K = _c(K, np.int8)
    V = _c(V, np.int8)
    ks = _c(ks, np.float32)
    vs = _c(vs, np.float32)
    D = q_code.size
    s, n = _sel_args(sel)
    out = np.zeros(D, np.float64)
    dropped = C.c_double()
    lib().orc_attend_int8_sv(D, L, blk, _ptr(q_code), float(q_scale), float(scale), _ptr(K),
                             _ptr(V), _ptr(ks), _ptr(vs), _ptr(s), n, float(eps), _ptr(out),
                             C.byref(dropped))
    return out, dropped.value


def dequant_rows(dtype, rows, scales=None):
    """Stored cache rows as binary64 values (every product is exact in binary64):
    f16 as is; int8 codes times their row's f32 scale; q8_0 codes times their
    32-channel group's f16 scale; q4_0 4-bit codes less 8 times that scale (the
    low nibble of byte i is channel 2i, the high nibble channel 2i + 1)."""
    rows = np.asarray(rows)
    if dtype == F16:
        return rows.astype(np.float16).astype(np.float64)
    if dtype == INT8:
        return rows.astype(np.float64) * np.asarray(scales, np.float32).astype(np.float64)[..., None]
    if dtype == Q4_0:
        r = rows.astype(np.int64)
        codes = np.empty(rows.shape[:-1] + (rows.shape[-1] * 2,), np.float64)
        codes[..., 0::2] = (r & 15) - 8
        codes[..., 1::2] = (r >> 4) - 8
    else:
        codes = rows.astype(np.float64)
    d = np.asarray(scales, np.float16).astype(np.float64)
    return codes * np.repeat(d, QGROUP, axis=-1)


def block_moments(X, blk):
    """Float16 means of the blocks of rows X [L, D] (binary64): [ceil(L / blk), D]."""
    X = _c(X, np.float64)
    L, D = X.shape
    nb = (L + blk - 1) // blk
    mean = np.zeros((max(nb, 1), D), np.uint16)
    lib().orc_block_moments(D, L, blk, _ptr(X), _ptr(mean))
    return mean[:nb].view(np.float16)


def attend_tail(q_exact, q_tail, K, V, L, blk, scale, sel, mK, mV):
    """Exact attention over the listed blocks plus the moment tail of every other
    block of [0, L): out [D] binary64.  K, V: [L, D] binary64 rows; mK, mV: the
    float16 block means."""
    q_exact = _c(q_exact, np.float64)
    q_tail = _c(q_tail, np.float64)
    K = _c(K, np.float64)
    V = _c(V, np.float64)
    mK = _c(mK, np.float16)
    mV = _c(mV, np.float16)
    D = q_exact.size
    s, n = _sel_args(np.zeros(0, np.int32) if sel is None else sel)
    out = np.zeros(D, np.float64)
    lib().orc_attend_tail(D, L, blk, _ptr(q_exact), _ptr(q_tail), float(scale), _ptr(K),
                          _ptr(V), _ptr(s), max(n, 0), _ptr(mK), _ptr(mV), _ptr(out))
    return out


def threads_available() -> int:
    return lib().orc_num_threads_available()


__all__ = ["F16", "INT8", "OracleCache", "half_to_double", "quantize_row", "block_scores",
           "forced_range", "select", "attend_f16", "qk_int8", "attend_int8", "attend_dequant",
           "sparse_v_keep", "attend_f16_sv", "attend_int8_sv", "Q8_0", "QGROUP",
           "double_to_half", "quantize_group32", "attend_q8_0", "Q4_0", "quantize_q4_0",
           "attend_q4_0", "dequant_rows", "block_moments", "attend_tail", "double_to_half_dir",
           "threads_available", "lib"]
