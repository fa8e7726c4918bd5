"""Host logic of bench.py: byte model, clock parsing, and the max-over-ranks
reduction on two gloo ranks (CPU, no GPU)."""
import os
import socket

import numpy as np
import torch.multiprocessing as mp

import bench
import workloads as W


def test_step_bytes_model():
    wl = W.WORKLOADS["llama2-7b-10k"]
    lens = W.seq_lens(wl)
    bm = bench.step_bytes(wl, lens, wl.modes)
    assert bm["kv"]["full"] == 160 * 2**20                 # 32 heads x 10240 x 512 B
    assert bm["kv"]["sparse"] == 8 * 2**20                 # 32 heads x 512 x 512 B
    assert bm["step_kv"] == 4 * 160 * 2**20 + 28 * 8 * 2**20
    tiny = W.WORKLOADS["tiny"]
    bt = bench.step_bytes(tiny, W.seq_lens(tiny), tiny.modes)
    assert bt["step_kv"] == 2 * 4 * 2**20 + 2 * 256 * 1024
    # ragged lengths shorter than k count only their own tokens
    short = tiny.with_(top_k=4096, max_seq_len=4096)
    assert bench.step_bytes(short, np.array([100]), [W.SPARSE])["kv"]["sparse"] == 100 * 2 * 512


def test_clock_summary_parses_nvidia_smi_rows():
    c = bench.ClockSampler(0)
    c.lines = [(1.0, "0, 1965, 2070, 800.1, 0x0, Not Active, Not Active, Not Active, Not Active"),
               (2.0, "0, 1980, 2070, 900.5, 0x4, Not Active, Not Active, Not Active, Active"),
               (2.5, "garbage"),
               (3.0, "0, 1200, 2070, 200.0, 0x1, Active, Not Active, Not Active, Not Active")]
    c.t_start, c.t_stop = 0.5, 2.9    # the last sample came after the timed region
    s = c.summary()
    assert s["sm_mhz"] == 1972.5 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"] and s["samples"] == 2
    c.t_stop = None                   # no stop mark: every sample from the start on counts
    s = c.summary()
    assert s["samples"] == 3 and s["reasons"] == ["hw_slowdown", "sw_power_cap"]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    bench.dist_init(world, "gloo")
    got = bench.dist_max(10.0 + rank * 5.5, world)
    bench.dist_barrier(world)
    q.put((rank, got))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_dist_max_over_two_gloo_ranks():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(2))
    assert res == {0: 15.5, 1: 15.5}


def test_single_rank_is_identity():
    assert bench.dist_max(3.25, 1) == 3.25


def test_traffic_records_follow_their_kernel_family(tmp_path, monkeypatch):
    """A committed DRAM-traffic record counts only while the sources of its
    own kernel family are unchanged: CUDA-core records are keyed to the
    CUDA-core sources, tensor-core records to the tensor-core ones."""
    assert bench.kernel_family("attention_kernel<1, 1, 0, 0, 0>") == "cuda"
    assert bench.kernel_family("attention_mma_ring_kernel<4>") == "mma"
    assert bench.kernel_family("attention_mma16_kernel<4, 0, 0, 0, 0>") == "mma"
    h_cuda, h_mma = bench.attn_source_hash("cuda"), bench.attn_source_hash("mma")
    assert h_cuda != h_mma and len(h_cuda) == len(h_mma) == 16
    rec = {
        "w:full": {"kernel": "attention_kernel<1, 0, 0, 0, 0>", "source_hash": h_cuda,
                   "dram_bytes_per_launch": 123},
        "w:sparse": {"kernel": "attention_mma_ring_kernel<4>", "source_hash": h_cuda,
                     "dram_bytes_per_launch": 456},  # keyed to the wrong family
        "v:sparse": {"kernel": "attention_mma_ring_kernel<4>", "source_hash": h_mma,
                     "dram_bytes_per_launch": 789},
    }
    f = tmp_path / "traffic.json"
    f.write_text(__import__("json").dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.measured_traffic("w", "full") == 123
    assert bench.measured_traffic("w", "sparse") is None
    assert bench.measured_traffic("v", "sparse") == 789
    assert bench.measured_traffic("v", "full") is None

