"""Seeded synthetic decode workloads (inputs only: no step of the method here).

Both the CUDA path and the CPU oracle read the tensors made here; this module
holds none of the method's arithmetic (no quantization, bound, selection or
softmax).  Shapes and value distributions follow the workloads the pages
measure: long single-token decode over a KV cache with grouped-query heads
(H query heads sharing Hkv KV heads, D = 128), keys with planted "needles"
that a retrieval query must find (the needle-in-a-haystack gate of the
"Quest-style block-selector" page, section "Correctness gate"), and int8
caches built from keys with a few outlier channels ("cpu-attn" card).

Every workload is drawn from a seeded ``torch.Generator`` on the device the
tensors are made on; the same seed gives the same tensors on the same device
type.  Keys and values are drawn in f32 and rounded to f16, the append input
format ``[B, n, Hkv, D]``; queries stay f32 ``[B, H, D]``.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

F16 = 0
INT8 = 1
Q8_0 = 2
Q4_0 = 3


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int                 # independent sequences
    H: int                 # query heads
    Hkv: int               # KV heads (GQA group G = H // Hkv)
    D: int                 # head dimension
    L: int                 # cached tokens
    dtype: int             # F16 or INT8 cache
    keys: str              # "iid" | "outliers" | "gqa_needles" | "drift_needles"
    k_sel: int             # top-K budget of non-forced blocks
    sink_tokens: int
    recent_tokens: int
    n_needles: int = 0     # needles per (sequence, KV head)
    seed: int = 1234
    block: int = 64

    @property
    def G(self) -> int:
        return self.H // self.Hkv

    @property
    def NB(self) -> int:
        return (self.L + self.block - 1) // self.block

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def coverage_budget(L: int, block: int, frac: float, sink: int, recent: int) -> int:
    """Top-K budget so that forced + top-K blocks make `frac` of all blocks."""
    nb = (L + block - 1) // block
    se = min(nb, (sink + block - 1) // block)
    rb = max(0, L - recent) // block if recent > 0 else nb
    forced = se + (nb - max(rb, se))
    return max(0, math.ceil(frac * nb) - forced)


# The five workloads of the decode study (sizes, distributions, budgets).
TINY = Workload("tiny_512_f16", B=1, H=8, Hkv=8, D=128, L=512, dtype=F16, keys="iid",
                k_sel=4, sink_tokens=4, recent_tokens=64, seed=1234)
INT8_DENSE = tuple(
    Workload(f"int8_dense_{L}", B=1, H=8, Hkv=8, D=128, L=L, dtype=INT8, keys="outliers",
             k_sel=0, sink_tokens=4, recent_tokens=64, seed=1235)
    for L in (512, 2048, 8192))
QWEN3_32K = Workload("qwen3_4b_gqa_32k_f16", B=1, H=32, Hkv=8, D=128, L=32768, dtype=F16,
                     keys="gqa_needles", n_needles=16, sink_tokens=4, recent_tokens=64,
                     k_sel=coverage_budget(32768, 64, 0.25, 4, 64), seed=1236)
CTX128K_B8 = Workload("ctx128k_b8_int8", B=8, H=32, Hkv=8, D=128, L=131072, dtype=INT8,
                      keys="gqa_needles", n_needles=16, sink_tokens=4, recent_tokens=256,
                      k_sel=131072 // 64 // 16, seed=1237)
CTX1M = Workload("ctx1m_int8", B=1, H=32, Hkv=8, D=128, L=1 << 20, dtype=INT8,
                 keys="drift_needles", n_needles=64, sink_tokens=4, recent_tokens=1024,
                 k_sel=1024, seed=1238)

# the 1M recipe on group-quantized (q8_0, q4_0) caches: same keys, same selection
CTX1M_Q8 = CTX1M.with_(name="ctx1m_q8_0", dtype=Q8_0)
CTX1M_Q4 = CTX1M.with_(name="ctx1m_q4_0", dtype=Q4_0)

WORKLOADS = {w.name: w for w in (TINY, *INT8_DENSE, QWEN3_32K, CTX128K_B8, CTX1M, CTX1M_Q8,
                                 CTX1M_Q4)}


def context_sweep(frac: float = 0.25):
    """The 32K GQA recipe (f16, per-head mean offsets, 16 needles) at 16K..1M
    context, each at `frac` block coverage (forced blocks included)."""
    out = []
    for L in (16384, 32768, 131072, 1 << 20):
        k_sel = coverage_budget(L, 64, frac, QWEN3_32K.sink_tokens, QWEN3_32K.recent_tokens)
        out.append(QWEN3_32K.with_(name=f"gqa_f16_{L // 1024}k_cov{round(frac * 100)}", L=L,
                                   k_sel=k_sel))
    return out


def head_dim_sweep(frac: float = 0.25, L: int = 131072):
    """The 32K GQA recipe at 128K context with head dims 64, 96, 128 and 256,
    on f16 and int8 caches, each at `frac` block coverage.  Head dim 128
    runs the tuned kernels, the others the general ones."""
    k_sel = coverage_budget(L, 64, frac, QWEN3_32K.sink_tokens, QWEN3_32K.recent_tokens)
    out = []
    for dtype, dn in ((F16, "f16"), (INT8, "int8")):
        for D in (64, 96, 128, 256):
            out.append(QWEN3_32K.with_(name=f"gqa_{dn}_128k_d{D}_cov{round(frac * 100)}", L=L,
                                       D=D, dtype=dtype, k_sel=k_sel))
    return out


def coverage_sweep():
    """The 128K x 8 int8 recipe with K_SEL = NB * c, c = 1/64 .. 1/2 (plus the
    sink and recent blocks)."""
    nb = CTX128K_B8.NB
    return [CTX128K_B8.with_(name=f"ctx128k_b8_int8_c1_{d}", k_sel=nb // d)
            for d in (64, 32, 16, 8, 4, 2)]


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_query(w: Workload, device="cpu", seed: Optional[int] = None) -> torch.Tensor:
    """q ~ N(0, 1), f32 [B, H, D]."""
    g = _gen(device, (w.seed if seed is None else seed) * 2 + 1)
    return torch.randn(w.B, w.H, w.D, generator=g, device=device, dtype=torch.float32)


def make_kv(w: Workload, q: torch.Tensor, device="cpu", chunk: int = 1 << 16):
    """Keys and values for the whole context, f16 [B, L, Hkv, D] each.

    Returns (k, v, needles) where needles is an int64 tensor [B, Hkv, n_needles]
    of planted token positions (empty when the recipe plants none).

    Recipes:
      iid            k, v ~ N(0, 1)
      outliers       iid, then round(1% of Hkv*D) (KV head, channel) slots
                     drawn from the seed are multiplied by 8 in k and v
      gqa_needles    k ~ N(0, 1) + mu[b, kvh] with mu ~ N(0, 1)^D fixed per
                     (sequence, KV head); n_needles positions per (sequence,
                     KV head) get k = 4 sqrt(D) * qhat, qhat the unit mean
                     direction of the group's query heads
      drift_needles  k ~ N(0, 1) + w_t with w a per-(sequence, KV head,
                     channel) random walk of N(0, 0.01^2) steps, plus needles
                     as above
    """
    B, L, Hkv, D = w.B, w.L, w.Hkv, w.D
    g = _gen(device, w.seed * 2)
    k = torch.empty(B, L, Hkv, D, dtype=torch.float16, device=device)
    v = torch.empty(B, L, Hkv, D, dtype=torch.float16, device=device)
    mu = None
    if w.keys == "gqa_needles":
        mu = torch.randn(B, 1, Hkv, D, generator=g, device=device)
    out_mask = None
    if w.keys == "outliers":
        n_out = round(0.01 * Hkv * D)
        slots = torch.randperm(Hkv * D, generator=g, device=device)[:n_out]
        out_mask = torch.ones(Hkv * D, device=device)
        out_mask[slots] = 8.0
        out_mask = out_mask.view(1, 1, Hkv, D)
    walk = torch.zeros(B, 1, Hkv, D, device=device) if w.keys == "drift_needles" else None
    for s in range(0, L, chunk):
        n = min(chunk, L - s)
        kc = torch.randn(B, n, Hkv, D, generator=g, device=device)
        vc = torch.randn(B, n, Hkv, D, generator=g, device=device)
        if mu is not None:
            kc += mu
        if out_mask is not None:
            kc *= out_mask
            vc *= out_mask
        if walk is not None:
            steps = torch.randn(B, n, Hkv, D, generator=g, device=device) * 0.01
            steps = torch.cumsum(steps, dim=1) + walk
            walk = steps[:, -1:].clone()
            kc += steps
        k[:, s:s + n] = kc.to(torch.float16)
        v[:, s:s + n] = vc.to(torch.float16)
    needles = torch.empty(B, Hkv, 0, dtype=torch.int64, device=device)
    if w.n_needles > 0:
        G = w.G
        qhat = q.view(B, Hkv, G, D).mean(dim=2)
        qhat = qhat / qhat.norm(dim=-1, keepdim=True)
        nk = (4.0 * math.sqrt(D) * qhat).to(torch.float16)     # [B, Hkv, D]
        pos = torch.stack([
            torch.stack([torch.randperm(L, generator=g, device=device)[:w.n_needles]
                         for _ in range(Hkv)]) for _ in range(B)])
        pos, _ = torch.sort(pos, dim=-1)
        for b in range(B):
            for h in range(Hkv):
                k[b, pos[b, h], h] = nk[b, h]
        needles = pos
    return k, v, needles


def make_step_token(w: Workload, step: int, device="cpu"):
    """The new token's k, v for one decode step, f16 [B, 1, Hkv, D] each."""
    g = _gen(device, w.seed * 7919 + step)
    k = torch.randn(w.B, 1, w.Hkv, w.D, generator=g, device=device).to(torch.float16)
    v = torch.randn(w.B, 1, w.Hkv, w.D, generator=g, device=device).to(torch.float16)
    return k, v


def make_workload(w: Workload, device="cpu"):
    q = make_query(w, device)
    k, v, needles = make_kv(w, q, device)
    return q, k, v, needles
