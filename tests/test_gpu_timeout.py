"""Failure detection without a GPU fault: a bounded device wait that nothing
ends gives up after its limit, records KVD_ERR_TIMEOUT in the status word, and
leaves the context usable (the kernels' own waits take the same path after
2 s).  No trap, device assert or endless loop is involved.
"""
import time

import pytest
import torch

import long_context_decode_kv_gb300 as kvd
from gpu_util import assert_outputs, dev, make_pair, scale_for, seeded

pytestmark = pytest.mark.gpu


def test_wait_runs_out_and_is_reported():
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    kvd.debug_wait_timeout(status, 20000)  # 20 ms
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert kvd.STATUS[int(status.item())] == "KVD_ERR_TIMEOUT"
    assert 0.019 <= elapsed < 5.0


def test_first_code_is_kept():
    status = torch.full((1,), 1, dtype=torch.int32, device=dev())  # KVD_ERR_INVALID already
    kvd.debug_wait_timeout(status, 1000)
    torch.cuda.synchronize()
    assert int(status.item()) == 1


def test_context_usable_after_a_timeout():
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    kvd.debug_wait_timeout(status, 5000)
    torch.cuda.synchronize()
    assert int(status.item()) == 5
    # the same stream and context run a decode that matches the oracle
    B, Hkv, G, L = 1, 2, 4, 700
    k = seeded((B, L, Hkv, 128), 901)
    v = seeded((B, L, Hkv, 128), 902)
    gc, oc = make_pair(kvd.INT8, k, v)
    q = seeded((B, Hkv * G, 128), 903, dtype=torch.float32)
    ws = kvd.make_workspace(gc, Hkv * G)
    out = torch.empty(B, Hkv * G, 128, device=dev())
    kvd.decode_attn_dense(gc, q, scale_for(), out, ws)
    torch.cuda.synchronize()
    ref, _, _ = oc.decode(q.cpu().numpy(), scale_for(), dense=True)
    assert_outputs(out, ref, kvd.INT8, "after timeout")
    assert gc.device_status() == 0
