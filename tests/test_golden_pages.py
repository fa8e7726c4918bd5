"""Values printed on the TidalDecode review page, checked against the
workload definitions and byte model that the bench and tests use."""
import os

import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def test_kv_cache_size_example():
    for layers, heads, dim, tokens, nbytes, want in _rows("kv_cache_size.txt"):
        got = W.kv_cache_bytes(int(layers), int(heads), int(dim), int(tokens), int(nbytes))
        assert got == int(want) == 64 * 2**30


def test_figure2_schedule():
    code = {W.FULL: "F", W.FULL_SELECT: "S", W.SPARSE: "P"}
    for family, layers, middle, modes in _rows("figure2_schedule.txt"):
        got = "".join(code[m] for m in W.figure2_schedule(int(layers), int(middle)))
        assert got == modes, family
        assert W.RESELECTION_LAYER[family] == int(middle)


def test_reselection_table_matches_workloads():
    table = {m: int(l) for m, l in _rows("reselection_layers.txt")}
    assert table["LLaMA-2-7B-LongChat"] == W.RESELECTION_LAYER["llama-2-7b"]
    assert table["LLaMA-3-8B"] == W.RESELECTION_LAYER["llama-3-8b"]
    sched = W.WORKLOADS["llama2-7b-10k"].modes
    assert sched[table["LLaMA-2-7B-Yarn"]] == W.FULL_SELECT
    sched = W.WORKLOADS["llama3-8b-32k"].modes
    assert sched[table["LLaMA-3.1-8B"]] == W.FULL_SELECT


def test_workload_table_shapes():
    tiny = W.WORKLOADS["tiny"]
    assert (tiny.q_heads, tiny.kv_heads, tiny.max_seq_len, tiny.top_k) == (8, 2, 4096, 256)
    assert tiny.modes == (W.FULL, W.FULL_SELECT, W.SPARSE, W.SPARSE)
    c4 = W.WORKLOADS["llama2-7b-100k"]
    assert W.kv_cache_bytes(c4.layers, c4.kv_heads, c4.head_dim, c4.max_seq_len) == 50 * 2**30
