"""Host logic of bench.py on CPU: the max-over-ranks and barrier used by the
multi-process run (gloo, world size 2), the launch count it claims per step,
and the reading of the committed traffic summary."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from long_context_decode_kv_gb300 import synth  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        m = bench.max_over_ranks(10.0 + 3.5 * rank, world)
        with open(os.path.join(out_dir, f"r{rank}"), "w") as f:
            f.write(repr(m))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2(tmp_path):
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, str(tmp_path))) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert [float(open(tmp_path / f"r{r}").read()) for r in range(2)] == [13.5, 13.5]


def test_single_rank_is_identity():
    assert bench.max_over_ranks(7.25, 1) == 7.25


@pytest.mark.parametrize("name,want", [("ctx1m_int8", 2), ("ctx128k_b8_int8", 2),
                                       ("tiny_512_f16", 2), ("int8_dense_2048", 3)])
def test_launches_per_step(name, want):
    # a top-K to rank with a recent window: the token rides in the selection
    # kernel (selection + decode); K_SEL = 0: append, fill, decode
    w = synth.WORKLOADS[name]
    assert bench.launches_per_step(w, w.L + 1) == want
    # nothing to rank once K_SEL covers every candidate
    assert bench.launches_per_step(w.with_(k_sel=10 ** 9), w.L + 1) == 3


def test_traffic_scaled_per_token(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "decode_kernel_traffic.txt").write_text(
        "# workload context digest dram_bytes tokens\n"
        "ctx1m_int8 262144 abc 1000 10\n"
        "ctx1m_int8 262144 old 9999 10\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_digest", lambda: "abc")
    assert bench.measured_traffic("ctx1m_int8", 25) == 2500.0
    assert bench.measured_traffic("ctx128k_b8_int8", 25) is None
    monkeypatch.setattr(bench, "source_digest", lambda: "new")
    assert bench.measured_traffic("ctx1m_int8", 25) is None


def test_committed_traffic_lines_are_well_formed():
    # every data line: a known workload, its context, a 16-hex-digit source
    # digest, and positive byte and token counts; each cited summary exists
    path = os.path.join(ROOT, "profiles", "decode_kernel_traffic.txt")
    seen = set()
    for line in open(path):
        if line.startswith("#"):
            for word in line.split():
                if word.startswith("profiles/") and word.endswith(".md"):
                    assert os.path.exists(os.path.join(ROOT, word)), word
            continue
        parts = line.split()
        if not parts:
            continue
        assert len(parts) == 5, line
        name, ctx, digest, nbytes, tokens = parts
        assert name in synth.WORKLOADS and name not in seen, name
        seen.add(name)
        assert int(ctx) > 0 and int(nbytes) > 0 and int(tokens) > 0
        assert len(digest) == 16 and int(digest, 16) >= 0
        # DRAM traffic at least the rows the tokens need: no impossible capture
        w = synth.WORKLOADS[name]
        assert int(nbytes) >= int(tokens) * bench.kv_bytes_per_token(w.dtype, w.D)
    assert "ctx1m_int8" in seen


def test_oracle_baseline_uses_every_core_it_can():
    # the all-core oracle leg spreads sequence 0's (KV head, query head)
    # attentions over the threads of this process's CPU affinity
    w = synth.QWEN3_32K.with_(L=2048, k_sel=8)
    q, k, v, _ = synth.make_workload(w, device="cpu")
    value, base = bench.oracle_leg_all_cores(w, q, k, v, 1)
    assert value > 0
    assert base["threads_available"] == len(os.sched_getaffinity(0))
    assert base["cores"] == min(len(os.sched_getaffinity(0)), w.Hkv * w.G)
