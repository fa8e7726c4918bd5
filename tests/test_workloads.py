"""The seeded generators: determinism, shapes, and that planting works."""
import numpy as np
import torch

import oracle
import workloads as W


def test_generate_is_deterministic():
    wl = W.WORKLOADS["tiny"]
    a = W.generate_layer(wl, 1)
    b = W.generate_layer(wl, 1)
    for x, y in zip(a, b):
        assert x.dtype == torch.bfloat16 and torch.equal(x, y)
    q, K, V = a
    assert q.shape == (1, 8, 128) and K.shape == (1, 2, 4096, 128) and V.shape == K.shape
    c = W.generate_layer(wl, 2)
    assert not torch.equal(a[1], c[1])


def test_heavy_sets_drift_and_bounds():
    wl = W.WORKLOADS["llama3-8b-32k"].with_(layers=4, max_seq_len=4096, heavy=100)
    sets = W.heavy_positions(wl)
    for s in sets:
        assert s.shape == (4, 8, 100)
        assert np.all(s >= 0) and np.all(s < 4096)
        for b in range(4):
            assert len(np.unique(s[b, 0])) == 100
            assert np.array_equal(s[b, 0], s[b, 7])       # shared by the sequence's heads
    kept = len(np.intersect1d(sets[0][0, 0], sets[1][0, 0]))
    assert kept == 80


def test_ragged_lengths_and_sinks():
    wl = W.WORKLOADS["serving-b32"]
    lens = W.seq_lens(wl)
    assert lens.shape == (32,) and lens.min() >= 8192 and lens.max() <= 16384
    c4 = W.WORKLOADS["llama2-7b-100k"].with_(layers=2, max_seq_len=2048, heavy=32)
    sets = W.heavy_positions(c4)
    assert np.all(sets[0] >= 4)


def test_planted_positions_are_enriched():
    """On a reduced LLaMA-2-shaped case the planted keys score about +1 above
    the rest (the recipe's bias of 1.0 along the shared direction), and the
    oracle's selection holds more of them than a random set would."""
    wl = W.WORKLOADS["llama2-7b-10k"].with_(layers=3, q_heads=2, kv_heads=2, max_seq_len=2048,
                                            heavy=64, top_k=64,
                                            modes=(W.FULL, W.FULL_SELECT, W.SPARSE))
    heavy = W.heavy_positions(wl)
    q, K, V = W.generate_layer(wl, 1, heavy=heavy[1])
    orc = oracle.get()
    gap, hits = [], 0
    for g in range(2):
        s = orc.group_scores(W.u16(q[0, g:g + 1]), W.u16(K[0, g]), 2048, oracle.scale_for(128))
        hv = heavy[1][0, g]
        rest = np.setdiff1d(np.arange(2048), hv)
        gap.append(s[hv].mean() - s[rest].mean())
        hits += len(np.intersect1d(orc.topk(s, 64), hv))
    assert np.mean(gap) > 0.4
    assert hits >= 3 * 2 * (64 * 64 / 2048)


def test_random_index_sets():
    idx = W.random_index_sets(3, 2, 2, 16, [10, 100], pad_fraction=0.25)
    assert np.all(idx[0, :, 10:] == -1)
    assert np.all(idx[1, :, :12] >= 0) and np.all(idx[1, :, 12:] == -1)
    for row in idx.reshape(-1, 16):
        live = row[row >= 0]
        assert np.all(np.diff(live) > 0)


def test_per_layer_select_schedule():
    assert W.per_layer_select_schedule(5) == (W.FULL, W.FULL, W.FULL_SELECT, W.FULL_SELECT,
                                              W.FULL_SELECT)
    assert W.per_layer_select_schedule(32).count(W.FULL_SELECT) == 30
