"""Whole decode steps through the C ABI (append one token, select, attend),
on device buffers and on host buffers, vs the oracle doing the same steps.
"""
import numpy as np
import pytest
import torch

import long_context_decode_kv_gb300 as kvd
from gpu_util import (assert_outputs, check_selection, dev, make_pair, oracle_attend_list,
                      scale_for, seeded)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", [kvd.F16, kvd.INT8, kvd.Q8_0, kvd.Q4_0])
@pytest.mark.parametrize("sparse", [True, False])
def test_steps_match_oracle(dtype, sparse):
    B, Hkv, G, L0, steps = 2, 2, 4, 1980, 6      # merges into block 30, then opens block 31
    k = seeded((B, L0, Hkv, 128), 141)
    v = seeded((B, L0, Hkv, 128), 142)
    gc, oc = make_pair(dtype, k, v, max_seq=2112)
    ws = kvd.make_workspace(gc, Hkv * G)
    k_sel, sink, recent = (7, 4, 64) if sparse else (-1, 0, 0)
    for s in range(steps):
        q = seeded((B, Hkv * G, 128), 150 + s, dtype=torch.float32)
        kn = seeded((B, 1, Hkv, 128), 160 + s)
        vn = seeded((B, 1, Hkv, 128), 170 + s)
        out = torch.empty(B, Hkv * G, 128, device=dev())
        sel_idx = torch.zeros((B, Hkv, gc.max_seq // 64), dtype=torch.int32, device=dev())
        sel_cnt = torch.zeros((B, Hkv), dtype=torch.int32, device=dev())
        kvd.decode_step(gc, q, kn, vn, scale_for(), k_sel, sink, recent, out, ws,
                        sel_idx=sel_idx if sparse else None, sel_cnt=sel_cnt if sparse else None)
        torch.cuda.synchronize()
        oc.append(kn.cpu().numpy(), vn.cpu().numpy())
        assert gc.len == oc.len == L0 + s + 1
        qn = q.cpu().numpy()
        if sparse:
            check_selection(sel_idx, sel_cnt, oc, qn, k_sel, sink, recent, G)
            # attend the GPU's own selection in the oracle (a tie swap, if
            # any, must not count against the attention kernel)
            ref = np.zeros((B, Hkv * G, 128))
            idx, cnt = sel_idx.cpu().numpy(), sel_cnt.cpu().numpy()
            for b in range(B):
                for g in range(Hkv):
                    ref[b, g * G:(g + 1) * G] = oracle_attend_list(
                        oc, qn[b, g * G:(g + 1) * G], b, g, idx[b, g, :cnt[b, g]], scale_for())
        else:
            ref, _, _ = oc.decode(qn, scale_for(), dense=True)
        assert_outputs(out, ref, dtype, f"step {s}")


@pytest.mark.parametrize("dtype", [kvd.F16, kvd.INT8, kvd.Q8_0, kvd.Q4_0])
@pytest.mark.parametrize("pinned", ["all", "none", "mixed"])
def test_host_step_equals_device_step(dtype, pinned):
    # pinned (device-mapped) host buffers are used in place by the kernels,
    # pageable ones are staged by copies; either way the step is the device one
    B, Hkv, G, L0 = 1, 8, 4, 5000
    k = seeded((B, L0, Hkv, 128), 181)
    v = seeded((B, L0, Hkv, 128), 182)
    a, _ = make_pair(dtype, k, v, max_seq=5120)
    b, _ = make_pair(dtype, k, v, max_seq=5120)
    wa = kvd.make_workspace(a, Hkv * G)
    wb = kvd.make_workspace(b, Hkv * G)
    for s in range(3):
        q = seeded((B, Hkv * G, 128), 190 + s, dtype=torch.float32)
        kn = seeded((B, 1, Hkv, 128), 195 + s)
        vn = seeded((B, 1, Hkv, 128), 199 + s)
        out_d = torch.empty(B, Hkv * G, 128, device=dev())
        kvd.decode_step(a, q, kn, vn, scale_for(), 20, 4, 128, out_d, wa)
        pin = {"all": (1, 1, 1, 1), "none": (0, 0, 0, 0), "mixed": (1, 0, 1, 0)}[pinned]
        qh, kh, vh = (t.cpu().pin_memory() if p else t.cpu().clone()
                      for t, p in zip((q, kn, vn), pin[:3]))
        out_h = torch.empty(B, Hkv * G, 128)
        out_h = out_h.pin_memory() if pin[3] else out_h
        kvd.decode_step_host(b, qh, kh, vh, scale_for(), 20, 4, 128, out_h, wb)
        torch.cuda.synchronize()
        assert torch.equal(out_d.cpu(), out_h)
    assert a.len == b.len == L0 + 3


def test_step_capacity_error_leaves_len():
    gc = kvd.KVCache(kvd.F16, 1, 1, 64, device=dev())
    k = seeded((1, 64, 1, 128), 5)
    kvd.kv_append(gc, k, k)
    ws = kvd.make_workspace(gc, 4)
    q = seeded((1, 4, 128), 6, dtype=torch.float32)
    out = torch.empty(1, 4, 128, device=dev())
    with pytest.raises(kvd.KvdError):
        kvd.decode_step(gc, q, k[:, :1].contiguous(), k[:, :1].contiguous(), 0.1, 2, 0, 0,
                        out, ws)
    assert gc.len == 64
