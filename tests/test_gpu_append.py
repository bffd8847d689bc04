"""GPU append (f16 copy / int8 or q8_0 absmax quantization + block envelope) vs the oracle.

Bar: cache rows, codes and scales bit-exact; bounds equal as numbers.
"""
import os

import numpy as np
import pytest
import torch

import long_context_decode_kv_gb300 as kvd
import oracle
from gpu_util import dev, make_pair, seeded

pytestmark = pytest.mark.gpu


def _compare(gc, oc):
    L = oc.len
    nb = (L + 63) // 64
    if gc.dtype == kvd.F16:
        assert torch.equal(gc.k[:, :, :L].cpu().view(torch.int16),
                           torch.from_numpy(oc.K[:, :, :L].view(np.int16)))
        assert torch.equal(gc.v[:, :, :L].cpu().view(torch.int16),
                           torch.from_numpy(oc.V[:, :, :L].view(np.int16)))
    elif gc.dtype in (kvd.Q8_0, kvd.Q4_0):
        assert np.array_equal(gc.k[:, :, :L].cpu().numpy(), oc.K[:, :, :L])
        assert np.array_equal(gc.v[:, :, :L].cpu().numpy(), oc.V[:, :, :L])
        assert np.array_equal(gc.k_scale[:, :, :L].cpu().numpy().view(np.uint16),
                              oc.kd[:, :, :L].view(np.uint16))
        assert np.array_equal(gc.v_scale[:, :, :L].cpu().numpy().view(np.uint16),
                              oc.vd[:, :, :L].view(np.uint16))
    else:
        assert np.array_equal(gc.k[:, :, :L].cpu().numpy(), oc.K[:, :, :L])
        assert np.array_equal(gc.v[:, :, :L].cpu().numpy(), oc.V[:, :, :L])
        assert np.array_equal(gc.k_scale[:, :, :L].cpu().numpy().view(np.uint32),
                              oc.ks[:, :, :L].view(np.uint32))
        assert np.array_equal(gc.v_scale[:, :, :L].cpu().numpy().view(np.uint32),
                              oc.vs[:, :, :L].view(np.uint32))
    assert np.array_equal(gc.kmin[:, :, :nb].cpu().float().numpy(),
                          oc.kmin[:, :, :nb].astype(np.float32))
    assert np.array_equal(gc.kmax[:, :, :nb].cpu().float().numpy(),
                          oc.kmax[:, :, :nb].astype(np.float32))


@pytest.mark.parametrize("dtype", [kvd.F16, kvd.INT8, kvd.Q8_0, kvd.Q4_0])
@pytest.mark.parametrize("L,chunks", [
    (1, None), (63, None), (64, None), (65, None), (300, None),
    (300, [1] * 70 + [230]), (1000, [63, 2, 64, 1, 870]), (4160, [4096, 1, 63]),
])
def test_append_matches_oracle(dtype, L, chunks):
    B, Hkv = 2, 3
    k = seeded((B, L, Hkv, 128), 100 + L)
    v = seeded((B, L, Hkv, 128), 200 + L)
    gc, oc = make_pair(dtype, k, v, chunks=chunks)
    _compare(gc, oc)


@pytest.mark.parametrize("dtype", [kvd.INT8, kvd.Q8_0, kvd.Q4_0])
@pytest.mark.parametrize("dist", ["outliers", "tiny", "ties", "zeros"])
def test_int8_quantization_edge_values(dist, dtype):
    B, L, Hkv = 1, 256, 2
    k = seeded((B, L, Hkv, 128), 7).float()
    v = seeded((B, L, Hkv, 128), 8).float()
    if dist == "outliers":
        k[..., 5] *= 8
        v[..., 77] *= 8
    elif dist == "tiny":
        k *= 1e-5
        v *= 3e-7  # f16 subnormals
    elif dist == "ties":
        # half-integer multiples of a power-of-two scale: exact .5 quotients
        g = torch.Generator(device=dev())
        g.manual_seed(3)
        k = torch.randint(-254, 255, k.shape, generator=g, device=dev()).float() / 2 * 0.25
        k[..., 0] = 127 * 0.25
        v = k.flip(-1)
    else:
        k[:, :10] = 0
        v[:, 5:20] = 0
    gc, oc = make_pair(dtype, k.half(), v.half())
    _compare(gc, oc)


def test_golden_quant_rows_through_append(golden_dir):
    rows = []
    for line in open(os.path.join(golden_dir, "quant_rows.txt")):
        line = line.strip()
        if not line or line.startswith("#") or "0x" in line:
            continue
        s, r, c = [x.strip() for x in line.split("|")]
        rows.append((float(s), [float(x) for x in r.split()], [int(x) for x in c.split()]))
    k = torch.zeros(1, len(rows), 1, 128)
    for i, (_, r, _) in enumerate(rows):
        k[0, i, 0, :len(r)] = torch.tensor(r)
    gc = kvd.KVCache(kvd.INT8, 1, 1, 64, device=dev())
    kh = k.half().to(dev())
    kvd.kv_append(gc, kh, kh.clone())
    torch.cuda.synchronize()
    for i, (s, r, c) in enumerate(rows):
        assert gc.k_scale[0, 0, i].item() == np.float32(s)
        assert gc.k[0, 0, i, :len(c)].cpu().tolist() == c


def test_append_capacity_and_len():
    gc = kvd.KVCache(kvd.F16, 1, 1, 64, device=dev())
    k = seeded((1, 65, 1, 128), 1)
    with pytest.raises(kvd.KvdError) as e:
        kvd.kv_append(gc, k, k)
    assert e.value.code == 3 and gc.len == 0
    kvd.kv_append(gc, k[:, :64].contiguous(), k[:, :64].contiguous())
    assert gc.len == 64


def test_bounds_merge_equals_recompute_over_many_small_appends():
    # 1-token decode appends across several blocks reproduce one-shot bounds
    B, L, Hkv = 1, 200, 2
    k = seeded((B, L, Hkv, 128), 11)
    v = seeded((B, L, Hkv, 128), 12)
    a, _ = make_pair(kvd.F16, k, v)
    b, _ = make_pair(kvd.F16, k, v, chunks=[1] * L)
    nb = 4
    assert torch.equal(a.kmin[:, :, :nb].float(), b.kmin[:, :, :nb].float())
    assert torch.equal(a.kmax[:, :, :nb].float(), b.kmax[:, :, :nb].float())


def _make_pair_f32(dtype, k, v, chunks, moments=False):
    B, L, Hkv, D = k.shape
    max_seq = (L + 64 + 63) // 64 * 64
    gc = kvd.KVCache(dtype, B, Hkv, max_seq, device=dev(), moments=moments)
    oc = oracle.OracleCache(dtype, B, Hkv, D, max_seq, 64)
    kh, vh = k.cpu().numpy(), v.cpu().numpy()
    s = 0
    for n in chunks:
        kvd.kv_append_f32(gc, k[:, s:s + n].contiguous(), v[:, s:s + n].contiguous())
        oc.append_f32(kh[:, s:s + n], vh[:, s:s + n])
        s += n
    torch.cuda.synchronize()
    assert gc.len == oc.len == L
    return gc, oc


@pytest.mark.parametrize("dtype", [kvd.F16, kvd.INT8, kvd.Q8_0, kvd.Q4_0])
@pytest.mark.parametrize("chunks", [[300], [1] * 70 + [230], [63, 2, 64, 1, 170]])
def test_append_f32_matches_oracle(dtype, chunks):
    # f32 input: rows, codes, scales and the outward-rounded bounds bit-exact
    B, Hkv, L = 2, 3, sum(chunks)
    k = seeded((B, L, Hkv, 128), 900, scale=3.0, dtype=torch.float32)
    v = seeded((B, L, Hkv, 128), 901, dtype=torch.float32)
    k[0, :5, 0, :4] = torch.tensor([1e-6, -1e-6, 3e4, -7e4])  # subnormal, large, past f16
    gc, oc = _make_pair_f32(dtype, k, v, chunks)
    _compare(gc, oc)


def test_append_f32_f16_cache_equals_f16_input():
    # the f16 cache stores the nearest f16 of each f32 value: the same cache as
    # appending those f16 values
    B, Hkv, L = 1, 2, 200
    k = seeded((B, L, Hkv, 128), 910, scale=2.0, dtype=torch.float32)
    v = seeded((B, L, Hkv, 128), 911, dtype=torch.float32)
    a = kvd.KVCache(kvd.F16, B, Hkv, 256, device=dev())
    b = kvd.KVCache(kvd.F16, B, Hkv, 256, device=dev())
    kvd.kv_append_f32(a, k, v)
    kvd.kv_append(b, k.half(), v.half())
    torch.cuda.synchronize()
    for name in ("k", "v", "kbounds"):
        assert torch.equal(getattr(a, name)[:, :, :L].view(torch.int16),
                           getattr(b, name)[:, :, :L].view(torch.int16)), name
