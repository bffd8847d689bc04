"""The GPU tests' comparison helper, pinned on the host: the oracle's
attention over a given block list (used to compare the GPU's output on the
GPU's own selection) equals the oracle's own decode step when the list is
the oracle's selection, for every cache type.  No GPU needed."""
import numpy as np
import pytest

import long_context_decode_kv_gb300 as kvd
import oracle
from gpu_util import oracle_attend_list


@pytest.mark.parametrize("dtype", [kvd.F16, kvd.INT8, kvd.Q8_0, kvd.Q4_0])
def test_oracle_attend_list_equals_decode(dtype):
    rng = np.random.default_rng(7 + dtype)
    B, Hkv, G, D, L = 2, 2, 4, 128, 700
    k = rng.standard_normal((B, L, Hkv, D)).astype(np.float16)
    v = rng.standard_normal((B, L, Hkv, D)).astype(np.float16)
    q = rng.standard_normal((B, Hkv * G, D)).astype(np.float32)
    oc = oracle.OracleCache(dtype, B, Hkv, D, 768, 64)
    oc.append(k, v)
    scale = 0.09
    ref, idx, cnt = oc.decode(q, scale, k_sel=3, sink_tokens=4, recent_tokens=64)
    for b in range(B):
        for g in range(Hkv):
            sel = idx[b, g, :cnt[b, g]]
            got = oracle_attend_list(oc, q[b, g * G:(g + 1) * G], b, g, sel, scale)
            assert np.array_equal(got, ref[b, g * G:(g + 1) * G])
            # a different list gives a different result (the list is used)
            other = oracle_attend_list(oc, q[b, g * G:(g + 1) * G], b, g, sel[1:], scale)
            assert not np.allclose(other, got)
