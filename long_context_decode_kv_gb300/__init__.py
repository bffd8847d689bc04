"""GB300-native Quest-style sparse decode attention over a long KV cache.

Thin Python binding over ``libkvdecode.so`` (C ABI in ``include/kvdecode.h``).
Every call marshals torch tensors to raw pointers and calls the library on the
tensor's CUDA stream; all arithmetic runs in the library's CUDA kernels.
PyTorch only provides device memory, streams and events.  There is no CPU
fallback: if the library is not built, loading it raises.

Entry points (same names as the C ABI, without the ``kvd_`` prefix):
  kv_append, select_blocks, decode_attn, decode_attn_dense, decode_step,
  decode_step_host, workspace_bytes, selected_count, status_string,
  debug_qk_int8, debug_scores, decode_attn_static.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional

import torch

from . import synth  # noqa: F401  (seeded inputs; no method arithmetic)

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libkvdecode.so")

F16 = 0
INT8 = 1
Q8_0 = 2
Q4_0 = 3
BLOCK = 64
HEAD_DIM = 128

STATUS = {0: "KVD_OK", 1: "KVD_ERR_INVALID", 2: "KVD_ERR_UNSUPPORTED", 3: "KVD_ERR_CAPACITY",
          4: "KVD_ERR_CUDA", 5: "KVD_ERR_TIMEOUT", 6: "KVD_ERR_WORKSPACE"}

EXPORTS = ("kvd_kv_append", "kvd_select_blocks", "kvd_decode_attn", "kvd_decode_attn_dense",
           "kvd_decode_step", "kvd_decode_step_host", "kvd_workspace_bytes",
           "kvd_selected_count", "kvd_status_string", "kvd_abi_version", "kvd_debug_qk_int8",
           "kvd_debug_scores", "kvd_decode_attn_static", "kvd_decode_attn_sv",
           "kvd_decode_attn_tail", "kvd_kv_append_f32", "kvd_select_blocks_per_head",
           "kvd_decode_attn_per_head", "kvd_debug_wait_timeout", "kvd_debug_stage_marks")


class KvdError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} -> {STATUS.get(code, code)}")


class CacheStruct(C.Structure):
    """Mirror of ``kvd_cache``."""
    _fields_ = [("dtype", C.c_int32), ("batch", C.c_int32), ("n_kv_heads", C.c_int32),
                ("head_dim", C.c_int32), ("max_seq", C.c_int32), ("block", C.c_int32),
                ("len", C.c_int32), ("reserved", C.c_int32),
                ("k", C.c_void_p), ("v", C.c_void_p), ("k_scale", C.c_void_p),
                ("v_scale", C.c_void_p), ("kbounds", C.c_void_p), ("dev_status", C.c_void_p),
                ("moments", C.c_void_p), ("seq_lens", C.c_void_p)]


_lib = None


def lib():
    """Load libkvdecode.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "long_context_decode_kv_gb300.build.build()")
        L = C.CDLL(LIB_PATH)
        p, i32, sz = C.c_void_p, C.c_int32, C.c_size_t
        cp = C.POINTER(CacheStruct)
        L.kvd_kv_append.argtypes = [cp, p, p, i32, p]
        L.kvd_kv_append_f32.argtypes = [cp, p, p, i32, p]
        L.kvd_select_blocks.argtypes = [cp, p, i32, i32, i32, i32, p, p, p, sz, p]
        L.kvd_decode_attn.argtypes = [cp, p, i32, C.c_float, p, p, i32, p, p, sz, p]
        L.kvd_decode_attn_dense.argtypes = [cp, p, i32, C.c_float, p, p, sz, p]
        L.kvd_decode_attn_static.argtypes = [cp, p, i32, C.c_float, p, p, i32, p, p]
        L.kvd_decode_attn_sv.argtypes = [cp, p, i32, C.c_float, p, p, i32, C.c_float, p, p, sz,
                                         p]
        L.kvd_select_blocks_per_head.argtypes = [cp, p, i32, i32, i32, i32, p, p, p, sz, p]
        L.kvd_decode_attn_per_head.argtypes = [cp, p, i32, C.c_float, p, p, i32, p, p, sz, p]
        L.kvd_decode_attn_tail.argtypes = [cp, p, i32, C.c_float, p, p, i32, p, p, sz, p]
        L.kvd_decode_step.argtypes = [cp, p, p, p, i32, C.c_float, i32, i32, i32, p, p, p, p,
                                      sz, p]
        L.kvd_decode_step_host.argtypes = [cp, p, p, p, i32, C.c_float, i32, i32, i32, p, p, p,
                                           p, sz, p]
        L.kvd_workspace_bytes.argtypes = [cp, i32]
        L.kvd_workspace_bytes.restype = sz
        L.kvd_selected_count.argtypes = [i32, i32, i32, i32, i32]
        L.kvd_selected_count.restype = i32
        L.kvd_status_string.argtypes = [i32]
        L.kvd_status_string.restype = C.c_char_p
        L.kvd_abi_version.restype = i32
        L.kvd_debug_qk_int8.argtypes = [cp, p, i32, p, p, p, p]
        L.kvd_debug_scores.argtypes = [cp, p, i32, p, p]
        L.kvd_debug_wait_timeout.argtypes = [p, i32, p]
        L.kvd_debug_stage_marks.argtypes = [p, sz]
        _lib = L
    return _lib


def _check(fn: str, rc: int):
    if rc != 0:
        raise KvdError(fn, rc)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return C.c_void_p(t.data_ptr())


def _stream(t: torch.Tensor, stream=None):
    if stream is None:
        stream = torch.cuda.current_stream(t.device)
    return C.c_void_p(stream.cuda_stream)


class KVCache:
    """Caller-owned cache tensors plus the C descriptor that points at them.

    k, v      [B, Hkv, max_seq, D]    float16 or int8 codes, or
              [B, Hkv, max_seq, D/2]  uint8 pairs of 4-bit codes (q4_0); D = head_dim:
              128, or any multiple of 16 up to 1024 for f16 / int8 caches without
              moments or seq_lens
    k_scale   [B, Hkv, max_seq]       float32 (int8), or
              [B, Hkv, max_seq, 4]    float16 group scales (q8_0, q4_0); same for v_scale
    kbounds   [B, Hkv, max_seq // 64, D, 2] float16: (kmin, kmax) per channel
    status    [1] int32 device word for device-side faults
    moments   [B, Hkv, max_seq // 64, 2, 128] float16 block means of K then V
              (only with moments=True: the moment tail of decode_attn_tail)
    seq_lens  optional [B] int32 device tensor of per-sequence lengths (each at
              most len; len is then the batch's maximum); see set_seq_lens
    """

    def __init__(self, dtype: int, batch: int, n_kv_heads: int, max_seq: int,
                 head_dim: int = HEAD_DIM, block: int = BLOCK, device="cuda",
                 tensors: Optional[dict] = None, moments: bool = False):
        self.dtype, self.batch, self.n_kv_heads = dtype, batch, n_kv_heads
        self.head_dim, self.max_seq, self.block = head_dim, max_seq, block
        dev = torch.device(device)
        if tensors is not None:
            self.t = dict(tensors)
        else:
            kvt = (torch.float16 if dtype == F16 else
                   torch.uint8 if dtype == Q4_0 else torch.int8)
            width = head_dim // 2 if dtype == Q4_0 else head_dim  # q4_0: two codes a byte
            nb = max_seq // block if block > 0 else 0
            self.t = {
                "k": torch.empty(batch, n_kv_heads, max_seq, width, dtype=kvt, device=dev),
                "v": torch.empty(batch, n_kv_heads, max_seq, width, dtype=kvt, device=dev),
                "kbounds": torch.empty(batch, n_kv_heads, nb, head_dim, 2, dtype=torch.float16,
                                       device=dev),
                "status": torch.zeros(1, dtype=torch.int32, device=dev),
            }
            if dtype == INT8:
                self.t["k_scale"] = torch.empty(batch, n_kv_heads, max_seq, dtype=torch.float32,
                                                device=dev)
                self.t["v_scale"] = torch.empty(batch, n_kv_heads, max_seq, dtype=torch.float32,
                                                device=dev)
            elif dtype in (Q8_0, Q4_0):
                ng = head_dim // 32
                self.t["k_scale"] = torch.empty(batch, n_kv_heads, max_seq, ng,
                                                dtype=torch.float16, device=dev)
                self.t["v_scale"] = torch.empty(batch, n_kv_heads, max_seq, ng,
                                                dtype=torch.float16, device=dev)
            if moments:
                self.t["moments"] = torch.empty(batch, n_kv_heads, nb, 2, head_dim,
                                                dtype=torch.float16, device=dev)
        self.s = CacheStruct(dtype, batch, n_kv_heads, head_dim, max_seq, block, 0, 0,
                             _ptr(self.t["k"]), _ptr(self.t["v"]),
                             _ptr(self.t.get("k_scale")), _ptr(self.t.get("v_scale")),
                             _ptr(self.t["kbounds"]), _ptr(self.t.get("status")),
                             _ptr(self.t.get("moments")))

    def set_seq_lens(self, seq_lens: Optional[torch.Tensor]):
        """Give every sequence its own length (an int32 [B] device tensor the
        caller owns and advances after each append), or None for one length."""
        if seq_lens is not None:
            assert seq_lens.dtype == torch.int32 and seq_lens.shape == (self.batch,)
            self.t["seq_lens"] = seq_lens
        else:
            self.t.pop("seq_lens", None)
        self.s.seq_lens = _ptr(seq_lens)

    def view(self, b: int) -> "KVCache":
        """Sequence b alone, as a batch-1 cache over the same memory (one
        sequence's rows, scales, bounds and means are contiguous slices)."""
        t = {k: v[b:b + 1] for k, v in self.t.items() if k not in ("status", "seq_lens")}
        t["status"] = self.t["status"]
        c = KVCache(self.dtype, 1, self.n_kv_heads, self.max_seq, self.head_dim, self.block,
                    device=self.t["k"].device, tensors=t)
        return c

    @property
    def kmin(self) -> torch.Tensor:
        """View [B, Hkv, max_seq // 64, 128] of the per-block channel minima."""
        return self.t["kbounds"][..., 0]

    @property
    def kmax(self) -> torch.Tensor:
        """View [B, Hkv, max_seq // 64, 128] of the per-block channel maxima."""
        return self.t["kbounds"][..., 1]

    @property
    def len(self) -> int:
        return self.s.len

    @len.setter
    def len(self, n: int):
        self.s.len = int(n)

    def __getattr__(self, name):
        t = self.__dict__.get("t")
        if t is not None and name in t:
            return t[name]
        raise AttributeError(name)

    def ref(self):
        return C.byref(self.s)

    def device_status(self) -> int:
        return int(self.t["status"].item())


def workspace_bytes(cache: KVCache, n_heads: int) -> int:
    return int(lib().kvd_workspace_bytes(cache.ref(), n_heads))


def make_workspace(cache: KVCache, n_heads: int) -> torch.Tensor:
    """A zero-filled, 256-byte aligned workspace for every call on this cache."""
    n = workspace_bytes(cache, n_heads)
    if n == 0:
        raise KvdError("kvd_workspace_bytes", 1)
    return torch.zeros(n, dtype=torch.uint8, device=cache.k.device)


def selected_count(length: int, k_sel: int, sink_tokens: int, recent_tokens: int,
                   block: int = BLOCK) -> int:
    return int(lib().kvd_selected_count(length, block, k_sel, sink_tokens, recent_tokens))


def status_string(code: int) -> str:
    return lib().kvd_status_string(code).decode()


def kv_append(cache: KVCache, k_new: torch.Tensor, v_new: torch.Tensor, stream=None):
    """k_new, v_new: [B, n_new, Hkv, D] float16 on the cache's device."""
    _check("kvd_kv_append", lib().kvd_kv_append(cache.ref(), _ptr(k_new), _ptr(v_new),
                                                int(k_new.shape[1]), _stream(k_new, stream)))


def kv_append_f32(cache: KVCache, k_new: torch.Tensor, v_new: torch.Tensor, stream=None):
    """k_new, v_new: [B, n_new, Hkv, D] float32 on the cache's device."""
    _check("kvd_kv_append_f32", lib().kvd_kv_append_f32(cache.ref(), _ptr(k_new), _ptr(v_new),
                                                        int(k_new.shape[1]),
                                                        _stream(k_new, stream)))


def select_blocks(cache: KVCache, q: torch.Tensor, k_sel: int, sink_tokens: int,
                  recent_tokens: int, sel_idx: torch.Tensor, sel_cnt: torch.Tensor,
                  workspace: torch.Tensor, stream=None):
    _check("kvd_select_blocks", lib().kvd_select_blocks(
        cache.ref(), _ptr(q), int(q.shape[1]), k_sel, sink_tokens, recent_tokens,
        _ptr(sel_idx), _ptr(sel_cnt), _ptr(workspace), workspace.numel(), _stream(q, stream)))


def decode_attn(cache: KVCache, q: torch.Tensor, softmax_scale: float, sel_idx: torch.Tensor,
                sel_cnt: torch.Tensor, max_sel: int, out: torch.Tensor,
                workspace: torch.Tensor, stream=None):
    _check("kvd_decode_attn", lib().kvd_decode_attn(
        cache.ref(), _ptr(q), int(q.shape[1]), float(softmax_scale), _ptr(sel_idx),
        _ptr(sel_cnt), int(max_sel), _ptr(out), _ptr(workspace), workspace.numel(),
        _stream(q, stream)))


def decode_attn_static(cache: KVCache, q: torch.Tensor, softmax_scale: float,
                       sel_idx: torch.Tensor, sel_cnt: torch.Tensor, max_sel: int,
                       out: torch.Tensor, stream=None):
    """decode_attn with no workspace: the scratch is a fixed array inside the
    library, shared by every call on the device (calls must not overlap)."""
    _check("kvd_decode_attn_static", lib().kvd_decode_attn_static(
        cache.ref(), _ptr(q), int(q.shape[1]), float(softmax_scale), _ptr(sel_idx),
        _ptr(sel_cnt), int(max_sel), _ptr(out), _stream(q, stream)))


def decode_attn_sv(cache: KVCache, q: torch.Tensor, softmax_scale: float, sel_idx,
                   sel_cnt, max_sel: int, sparse_v_eps: float, out: torch.Tensor,
                   workspace: torch.Tensor, stream=None):
    """decode_attn with sparse-V in eps mode; sel_idx None attends every block."""
    _check("kvd_decode_attn_sv", lib().kvd_decode_attn_sv(
        cache.ref(), _ptr(q), int(q.shape[1]), float(softmax_scale), _ptr(sel_idx),
        _ptr(sel_cnt), int(max_sel), float(sparse_v_eps), _ptr(out), _ptr(workspace),
        workspace.numel(), _stream(q, stream)))


def select_blocks_per_head(cache: KVCache, q: torch.Tensor, k_sel: int, sink_tokens: int,
                           recent_tokens: int, sel_idx: torch.Tensor, sel_cnt: torch.Tensor,
                           workspace: torch.Tensor, stream=None):
    """Selection per query head: sel_idx [B, H, max_seq // 64], sel_cnt [B, H] int32."""
    _check("kvd_select_blocks_per_head", lib().kvd_select_blocks_per_head(
        cache.ref(), _ptr(q), int(q.shape[1]), int(k_sel), int(sink_tokens),
        int(recent_tokens), _ptr(sel_idx), _ptr(sel_cnt), _ptr(workspace), workspace.numel(),
        _stream(q, stream)))


def decode_attn_per_head(cache: KVCache, q: torch.Tensor, softmax_scale: float, sel_idx,
                         sel_cnt, max_sel: int, out: torch.Tensor, workspace: torch.Tensor,
                         stream=None):
    """decode_attn over lists per query head (select_blocks_per_head's rows)."""
    _check("kvd_decode_attn_per_head", lib().kvd_decode_attn_per_head(
        cache.ref(), _ptr(q), int(q.shape[1]), float(softmax_scale), _ptr(sel_idx),
        _ptr(sel_cnt), int(max_sel), _ptr(out), _ptr(workspace), workspace.numel(),
        _stream(q, stream)))


def decode_attn_tail(cache: KVCache, q: torch.Tensor, softmax_scale: float, sel_idx, sel_cnt,
                     max_sel: int, out: torch.Tensor, workspace: torch.Tensor, stream=None):
    """decode_attn plus the moment tail of every block the lists leave out
    (needs a cache made with moments=True)."""
    _check("kvd_decode_attn_tail", lib().kvd_decode_attn_tail(
        cache.ref(), _ptr(q), int(q.shape[1]), float(softmax_scale), _ptr(sel_idx),
        _ptr(sel_cnt), int(max_sel), _ptr(out), _ptr(workspace), workspace.numel(),
        _stream(q, stream)))


def decode_attn_dense(cache: KVCache, q: torch.Tensor, softmax_scale: float, out: torch.Tensor,
                      workspace: torch.Tensor, stream=None):
    _check("kvd_decode_attn_dense", lib().kvd_decode_attn_dense(
        cache.ref(), _ptr(q), int(q.shape[1]), float(softmax_scale), _ptr(out),
        _ptr(workspace), workspace.numel(), _stream(q, stream)))


def decode_step(cache: KVCache, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                softmax_scale: float, k_sel: int, sink_tokens: int, recent_tokens: int,
                out: torch.Tensor, workspace: torch.Tensor, sel_idx=None, sel_cnt=None,
                stream=None):
    _check("kvd_decode_step", lib().kvd_decode_step(
        cache.ref(), _ptr(q), _ptr(k_new), _ptr(v_new), int(q.shape[1]), float(softmax_scale),
        k_sel, sink_tokens, recent_tokens, _ptr(sel_idx), _ptr(sel_cnt), _ptr(out),
        _ptr(workspace), workspace.numel(), _stream(workspace, stream)))


def decode_step_host(cache: KVCache, q_host: torch.Tensor, k_new_host: torch.Tensor,
                     v_new_host: torch.Tensor, softmax_scale: float, k_sel: int,
                     sink_tokens: int, recent_tokens: int, out_host: torch.Tensor,
                     workspace: torch.Tensor, sel_idx=None, sel_cnt=None, stream=None):
    """Host (ideally pinned) q/k_new/v_new in, host out; synchronize before reading out."""
    _check("kvd_decode_step_host", lib().kvd_decode_step_host(
        cache.ref(), _ptr(q_host), _ptr(k_new_host), _ptr(v_new_host), int(q_host.shape[1]),
        float(softmax_scale), k_sel, sink_tokens, recent_tokens, _ptr(sel_idx), _ptr(sel_cnt),
        _ptr(out_host), _ptr(workspace), workspace.numel(), _stream(workspace, stream)))


def debug_qk_int8(cache: KVCache, q: torch.Tensor, dots: torch.Tensor, q_codes: torch.Tensor,
                  q_scales: torch.Tensor, stream=None):
    _check("kvd_debug_qk_int8", lib().kvd_debug_qk_int8(
        cache.ref(), _ptr(q), int(q.shape[1]), _ptr(dots), _ptr(q_codes), _ptr(q_scales),
        _stream(q, stream)))


def debug_wait_timeout(status: torch.Tensor, limit_us: int, stream=None):
    """Run the bounded-wait path on a wait that nothing ends (status: int32 [1])."""
    _check("kvd_debug_wait_timeout", lib().kvd_debug_wait_timeout(
        _ptr(status), int(limit_us), _stream(status, stream)))


MARK_SLOTS = 16
MARK_CTAS = 4096
MARK_KINDS = 3


def debug_stage_marks(marks: Optional[torch.Tensor]):
    """Give the library a device buffer for stage marks (int64, at least
    MARK_KINDS * MARK_CTAS * MARK_SLOTS elements), or None to stop recording.
    Raises KvdError (UNSUPPORTED) unless the library was built with marks."""
    n = 0 if marks is None else marks.numel() * marks.element_size()
    _check("kvd_debug_stage_marks", lib().kvd_debug_stage_marks(_ptr(marks), n))


def debug_scores(cache: KVCache, q: torch.Tensor, ub: torch.Tensor, stream=None):
    _check("kvd_debug_scores", lib().kvd_debug_scores(
        cache.ref(), _ptr(q), int(q.shape[1]), _ptr(ub), _stream(q, stream)))


__all__ = ["F16", "INT8", "Q8_0", "Q4_0", "BLOCK", "HEAD_DIM", "KVCache", "KvdError", "CacheStruct", "lib",
           "debug_stage_marks", "MARK_SLOTS", "MARK_CTAS", "MARK_KINDS",
           "workspace_bytes", "make_workspace", "selected_count", "status_string", "kv_append",
           "kv_append_f32", "select_blocks", "decode_attn", "decode_attn_dense", "decode_attn_static",
           "decode_attn_sv", "decode_attn_tail", "select_blocks_per_head",
           "decode_attn_per_head", "decode_step",
           "decode_step_host", "debug_qk_int8", "debug_scores", "debug_wait_timeout", "synth", "EXPORTS"]
