"""CUDA path (through the C ABI) against the CPU oracle on the same seeded inputs.

Small cases span several splits and ragged tails and are compared element by
element; degenerate cases (empty context, k >= N, padding, ties) are covered
explicitly.  The full-size workloads live in test_parity_full_gpu.py.
"""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_td_gb300 as td
import workloads as W
from parity_util import check_index_set, check_outputs

pytestmark = pytest.mark.gpu
D = 128


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    td.td_set_tuning("max_splits", 0)


PATHS = {
    "streamed": {"full_staged": 0, "sparse_staged": 0, "mma": 0},
    "staged": {"full_staged": 1, "sparse_staged": 1, "mma": 0},
    "tma": {"full_staged": 1, "sparse_staged": 2, "mma": 0},
    "mma": {"mma": 1},
    "mma8": {"mma": 1, "mma_full_tokens": 8, "mma_sparse_tokens": 8, "full_prefetch": 2},
    "mma16": {"mma": 1, "mma_sparse_tokens": 16, "full_prefetch": 2},
    "mma32": {"mma": 1, "mma_full_tokens": 32, "mma_sparse_tokens": 32},
    "ring": {"mma": 1, "mma_sparse_tokens": 64},
    "chunked": {"mma": 1, "full_interleave": 0},
    "stream_k": {"mma": 1, "sparse_stream_k": 1},
}
TUNING_KEYS = ("full_staged", "sparse_staged", "mma", "full_prefetch", "mma_full_tokens",
               "mma_sparse_tokens", "sparse_stream_k", "full_interleave")


@pytest.fixture(scope="module", autouse=True, params=list(PATHS))
def staged(request):
    """Every case runs on each kernel path: CUDA-core kernels with
    register-streamed loads, the same with rows staged through shared memory
    (bulk copies for full layers; per-thread cp.async, or TMA row gathers, for
    sparse layers), and the tensor-core kernels (grouped-query layers with G = 4, 8; other
    groups keep the CUDA-core kernels) in three tilings: the default (16
    tokens per warp per round for full and full+select layers, the
    shared-memory ring for sparse layers), 8 tokens per warp for every layer
    kind, and 16 for every layer
    kind, these two also prefetching two rounds ahead into L2 on full layers
    (the default is one round); 16 tokens per warp with two rounds in
    flight per warp for every layer kind; sparse layers staged through a
    ring of shared-memory rounds read back by ldmatrix; and sparse layers
    under the stream-K partition (a 1D grid sharing the layer's rounds
    evenly)."""
    for key, value in PATHS[request.param].items():
        td.td_set_tuning(key, value)
    yield request.param
    for key in TUNING_KEYS:
        td.td_set_tuning(key, -1)


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


@pytest.fixture(params=[(1024, 0, 1), (512, 0, 1), (1024, 2048, 1), (1024, 0, 2), (1024, 0, 4),
                        (1024, 2048, 8)],
                ids=["t1024", "t512", "t1024-warp2048", "cluster2", "cluster4", "cluster8-warp2048"])
def topk_threads(request):
    """Both block sizes of the top-k kernel with one CTA per row, the
    threshold-bin select taken by one warp up to 2048 candidates instead of
    the default 256 (so the adversarial rows run through both select paths),
    and clusters of 2, 4 and 8 CTAs per row (each scanning a slice of the
    row, merged through distributed shared memory)."""
    threads, warp_max, cluster = request.param
    td.td_set_tuning("topk_threads", threads)
    td.td_set_tuning("topk_warp_max", warp_max)
    td.td_set_tuning("topk_cluster", cluster)
    yield threads
    td.td_set_tuning("topk_threads", 0)
    td.td_set_tuning("topk_warp_max", 0)
    td.td_set_tuning("topk_cluster", 0)


def _dev(*ts):
    return [t.cuda() for t in ts]


def run_full(shape, q, K, V, lens, top_k=0):
    B, Hq, Hkv = shape.batch, shape.num_q_heads, shape.num_kv_heads
    qd, Kd, Vd = _dev(q, K, V)
    seq = torch.as_tensor(np.asarray(lens, np.int32)).cuda()
    out = torch.empty_like(qd)
    out32 = torch.empty(qd.shape, dtype=torch.float32, device="cuda")
    idx = torch.full((B, Hkv, max(top_k, 1)), -7, dtype=torch.int32, device="cuda")
    scores = torch.full((B, Hkv, shape.max_seq_len), float("nan"), device="cuda")
    ws = td.Workspace(shape, top_k)
    td.td_full_attn_select(shape, qd, Kd, Vd, seq, top_k, idx if top_k else None, out, out32,
                           scores if top_k else None, ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    return out, out32, idx[..., :top_k].cpu().numpy(), scores.cpu().numpy()


def oracle_full(orc, shape, q, K, V, lens):
    B, Hq, Hkv = shape.batch, shape.num_q_heads, shape.num_kv_heads
    G = Hq // Hkv
    qb, Kb, Vb = W.u16(q), W.u16(K), W.u16(V)
    ref = np.zeros((B, Hq, D))
    for b in range(B):
        for h in range(Hq):
            ref[b, h] = orc.attend(qb[b, h], Kb[b, h // G, :lens[b]], Vb[b, h // G, :lens[b]],
                                   shape.scale)
    return ref


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("max_splits", [0, 1])
def test_full_attention_ragged(orc, G, max_splits):
    td.td_set_tuning("max_splits", max_splits)
    Hkv, B, N = 2, 4, 700
    lens = [700, 0, 333, 45]            # full, empty, ragged tail, shorter than one round
    shape = td.make_shape(B, G * Hkv, Hkv, N, scale=td.default_scale(D))
    q, K, V, _ = W.random_case(10 + G, B, G * Hkv, Hkv, N, lens)
    out, out32, _, _ = run_full(shape, q, K, V, lens)
    ref = oracle_full(orc, shape, q, K, V, lens)
    check_outputs(out, out32, ref, f"G={G}")
    assert torch.all(out[1] == 0) and torch.all(out32[1] == 0)   # empty context -> 0
    td.td_set_tuning("max_splits", 0)


def test_full_attention_planted_large_logits(orc):
    """Sink-like keys (x3) and planted directions give logits up to ~30."""
    wl = W.WORKLOADS["llama2-7b-100k"].with_(batch=1, layers=1, q_heads=4, kv_heads=4,
                                             max_seq_len=3000, heavy=64, top_k=128)
    q, K, V = W.generate_layer(wl, 0)
    shape = td.make_shape(1, 4, 4, 3000, scale=td.default_scale(D))
    out, out32, _, _ = run_full(shape, q, K, V, [3000])
    check_outputs(out, out32, oracle_full(orc, shape, q, K, V, [3000]), "planted")


@pytest.mark.parametrize("G,k", [(1, 64), (4, 100), (8, 256), (2, 1)])
def test_full_select_scores_and_sets(orc, G, k, topk_threads):
    Hkv, B, N = 2, 3, 1500
    lens = [1500, 777, 50]              # the last row has fewer tokens than k for k >= 64
    shape = td.make_shape(B, G * Hkv, Hkv, N, scale=td.default_scale(D))
    q, K, V, _ = W.random_case(20 + G, B, G * Hkv, Hkv, N, lens)
    out, out32, idx, scores = run_full(shape, q, K, V, lens, top_k=k)
    check_outputs(out, out32, oracle_full(orc, shape, q, K, V, lens), "select outputs")
    qb, Kb = W.u16(q), W.u16(K)
    exact = 0
    for b in range(B):
        for g in range(Hkv):
            s_ref = orc.group_scores(qb[b, g * G:(g + 1) * G], Kb[b, g], lens[b], shape.scale)
            s_got = scores[b, g, :lens[b]].astype(np.float64)
            assert np.allclose(s_got, s_ref, rtol=1e-5, atol=1e-4), "emitted scores off"
            assert np.all(np.isnan(scores[b, g, lens[b]:]))      # nothing written past N_b
            ref_idx = orc.topk(s_ref, k)
            exact += check_index_set(idx[b, g], ref_idx, s_ref, k, f"b{b} g{g}")
    assert exact >= B * Hkv - 1


def _topk_case(scores_rows, lens, k):
    """Run td_topk_select on explicit fp32 score rows ([B][1][Nmax])."""
    B = len(scores_rows)
    N = max(len(r) for r in scores_rows)
    arr = np.full((B, 1, N), 7.0, dtype=np.float32)
    for b, r in enumerate(scores_rows):
        arr[b, 0, :len(r)] = r
    shape = td.make_shape(B, 1, 1, N)
    sc = torch.as_tensor(arr).cuda()
    seq = torch.as_tensor(np.asarray(lens, np.int32)).cuda()
    idx = torch.full((B, 1, k), -9, dtype=torch.int32, device="cuda")
    ws = td.Workspace(shape, k)
    td.td_topk_select(shape, sc, seq, k, idx, ws)
    torch.cuda.synchronize()
    return arr, idx.cpu().numpy()


def test_topk_adversarial(orc, topk_threads):
    rs = np.random.RandomState(5)
    N = 5000
    rows = [
        rs.randn(N).astype(np.float32),                                  # random
        np.zeros(N, np.float32),                                         # all equal
        np.round(rs.randn(N) * 2).astype(np.float32),                    # many ties at the k-th
        np.where(rs.rand(N) < 0.5, -0.0, 0.0).astype(np.float32),        # +-0 only
        -np.abs(rs.randn(N)).astype(np.float32),                         # negative only
        np.concatenate([np.full(10, 3.0), np.full(N - 10, -1.0)]).astype(np.float32),
        np.array([np.inf, -np.inf, 1.0, -1.0] * (N // 4), np.float32),   # infinities
        rs.randn(N).astype(np.float32),                                  # N_b < k (lens 40)
        rs.randn(N).astype(np.float32),                                  # N_b = 0
        (rs.randint(0, 3, N) * 1e-39).astype(np.float32),                # subnormal ties
    ]
    lens = [N] * 7 + [40, 0, N]
    for k in (1, 64, 300, N):
        arr, got = _topk_case(rows, lens, k)
        for b in range(len(rows)):
            want = orc.topk(arr[b, 0, :lens[b]].astype(np.float64), k)
            assert np.array_equal(got[b, 0], want), f"row {b} k={k}"


def test_topk_large_rows(orc, topk_threads):
    rs = np.random.RandomState(6)
    N, k = 102400, 4096
    rows = [np.round(rs.randn(N) * 50).astype(np.float32) for _ in range(3)]
    lens = [N, N - 1, 65537]
    arr, got = _topk_case(rows, lens, k)
    for b in range(3):
        want = orc.topk(arr[b, 0, :lens[b]].astype(np.float64), k)
        assert np.array_equal(got[b, 0], want), f"row {b}"


def test_topk_rows_longer_than_the_bitmap(orc):
    """Rows up to 2^18 positions are written through a shared-memory bitmap;
    longer ones take the ordered-compaction path.  Lengths at, just past and
    well past the boundary, with heavy ties at the k-th score."""
    rs = np.random.RandomState(8)
    N = 300000
    rows = [rs.randn(N).astype(np.float32),
            np.round(rs.randn(N) * 4).astype(np.float32),
            np.round(rs.randn(N) * 4).astype(np.float32)]
    lens = [N, 1 << 18, (1 << 18) + 1]
    for k in (1, 4096, 100000):
        arr, got = _topk_case(rows, lens, k)
        for b in range(len(rows)):
            want = orc.topk(arr[b, 0, :lens[b]].astype(np.float64), k)
            assert np.array_equal(got[b, 0], want), f"row {b} k={k}"


def test_topk_threshold_bin_larger_than_shared_memory(orc, topk_threads):
    """More than 16384 (512-thread CTAs: 8192) scores share the threshold's
    top bits: the kernel's streaming fallback path (heavy ties at and around
    the k-th score)."""
    rs = np.random.RandomState(7)
    N = 60000
    rows = [np.zeros(N, np.float32),                                   # one bin, all tied
            rs.randint(0, 2, N).astype(np.float32),                    # two values
            (1.0 + rs.randint(0, 64, N) * 2.0 ** -20).astype(np.float32)]  # one 11-bit bin, 64 values
    lens = [N, N - 3, N]
    for k in (1, 1000, 30001):
        arr, got = _topk_case(rows, lens, k)
        for b in range(len(rows)):
            want = orc.topk(arr[b, 0, :lens[b]].astype(np.float64), k)
            assert np.array_equal(got[b, 0], want), f"row {b} k={k}"


def run_sparse(shape, q, K, V, lens, idx_np, top_k):
    qd, Kd, Vd = _dev(q, K, V)
    seq = torch.as_tensor(np.asarray(lens, np.int32)).cuda()
    idx = torch.as_tensor(idx_np.astype(np.int32)).cuda()
    out = torch.empty_like(qd)
    out32 = torch.empty(qd.shape, dtype=torch.float32, device="cuda")
    ws = td.Workspace(shape, top_k)
    td.td_sparse_attn(shape, qd, Kd, Vd, seq, idx, top_k, out, out32, ws)
    torch.cuda.synchronize()
    return out, out32, ws.status()


def oracle_sparse(orc, shape, q, K, V, idx_np):
    B, Hq, Hkv = shape.batch, shape.num_q_heads, shape.num_kv_heads
    G = Hq // Hkv
    qb, Kb, Vb = W.u16(q), W.u16(K), W.u16(V)
    ref = np.zeros((B, Hq, D))
    for b in range(B):
        for h in range(Hq):
            rows = idx_np[b, h // G]
            rows = rows[rows >= 0]
            ref[b, h] = orc.attend(qb[b, h], Kb[b, h // G], Vb[b, h // G], shape.scale, rows=rows)
    return ref


@pytest.mark.parametrize("G,k", [(1, 300), (4, 64), (8, 1000), (2, 1)])
def test_sparse_random_sets(orc, G, k):
    Hkv, B, N = 2, 3, 2000
    lens = [2000, 1200, 500]
    shape = td.make_shape(B, G * Hkv, Hkv, N, scale=td.default_scale(D))
    q, K, V, _ = W.random_case(30 + G, B, G * Hkv, Hkv, N, lens)
    idx = W.random_index_sets(31 + G, B, Hkv, k, lens, pad_fraction=0.1 if k > 1 else 0.0)
    rs = np.random.RandomState(32)
    for row in idx.reshape(-1, k):             # order inside a set must not matter
        rs.shuffle(row)
    out, out32, status = run_sparse(shape, q, K, V, lens, idx, k)
    assert status == 0
    check_outputs(out, out32, oracle_sparse(orc, shape, q, K, V, idx), f"sparse G={G} k={k}")


def test_sparse_all_padding_and_all_positions(orc):
    G, Hkv, B, N = 4, 2, 2, 640
    lens = [640, 640]
    shape = td.make_shape(B, G * Hkv, Hkv, N, scale=td.default_scale(D))
    q, K, V, _ = W.random_case(40, B, G * Hkv, Hkv, N, lens)
    idx = np.full((B, Hkv, N), -1, np.int32)
    idx[0] = np.arange(N)                      # k = N: every position
    out, out32, status = run_sparse(shape, q, K, V, lens, idx, N)
    assert status == 0
    assert torch.all(out[1] == 0)              # all padding -> 0
    fo, fo32, _, _ = run_full(shape, q, K, V, lens)
    ref = oracle_full(orc, shape, q, K, V, lens)
    check_outputs(out[:1], out32[:1], ref[:1], "k=N sparse")
    # sparse over every position equals full attention (fp32, different split order)
    assert torch.allclose(out32[0], fo32[0], rtol=0, atol=1e-5 * float(fo32[0].abs().max()))


def test_sparse_bad_index_is_flagged_and_skipped(orc):
    G, Hkv, B, N = 1, 1, 1, 256
    shape = td.make_shape(B, G * Hkv, Hkv, N, scale=td.default_scale(D))
    q, K, V, _ = W.random_case(41, B, 1, 1, N, [200])
    good = np.array([[[3, 50, 199, -1]]], np.int32)
    bad = np.array([[[3, 50, 199, 200]]], np.int32)     # 200 >= seq_lens[0]
    out_g, out32_g, st_g = run_sparse(shape, q, K, V, [200], good, 4)
    out_b, out32_b, st_b = run_sparse(shape, q, K, V, [200], bad, 4)
    assert st_g == 0 and st_b == td.FLAG_INDEX_OUT_OF_RANGE
    assert torch.equal(out32_g, out32_b)


def test_seq_len_out_of_range_is_flagged(orc):
    shape = td.make_shape(1, 2, 2, 128, scale=td.default_scale(D))
    q, K, V, _ = W.random_case(42, 1, 2, 2, 128, [128])
    qd, Kd, Vd = _dev(q, K, V)
    seq = torch.tensor([500], dtype=torch.int32, device="cuda")      # > max_seq_len
    out = torch.empty_like(qd)
    out32 = torch.empty(qd.shape, dtype=torch.float32, device="cuda")
    ws = td.Workspace(shape, 0)
    td.td_full_attn_select(shape, qd, Kd, Vd, seq, 0, None, out, out32, None, ws)
    assert ws.status() == td.FLAG_SEQ_LEN_OUT_OF_RANGE
    check_outputs(out, out32, oracle_full(orc, shape, q, K, V, [128]), "clamped")


def _tiny_inputs():
    wl = W.WORKLOADS["tiny"]
    heavy = W.heavy_positions(wl)
    layers = [W.generate_layer(wl, layer, "cpu", heavy[layer]) for layer in range(wl.layers)]
    return wl, layers


@pytest.mark.parametrize("schedule", ["figure2", "per_layer_select"])
def test_decode_step_tiny_matches_oracle(orc, schedule):
    wl, layers = _tiny_inputs()
    if schedule == "per_layer_select":     # selection at every layer after the first two
        wl = wl.with_(modes=W.per_layer_select_schedule(wl.layers))
    lens = W.seq_lens(wl)
    shape = td.make_shape(wl.batch, wl.q_heads, wl.kv_heads, wl.max_seq_len,
                          scale=td.default_scale(D))
    q = [x[0].cuda() for x in layers]
    K = [x[1].cuda() for x in layers]
    V = [x[2].cuda() for x in layers]
    outs = [torch.empty_like(x) for x in q]
    outs32 = [torch.empty(x.shape, dtype=torch.float32, device="cuda") for x in q]
    idx = torch.full((1, wl.kv_heads, wl.top_k), -1, dtype=torch.int32, device="cuda")
    ws = td.Workspace(shape, wl.top_k)
    td.td_decode_step(shape, wl.modes, q, K, V, torch.as_tensor(lens).cuda(), wl.top_k, idx,
                      outs, outs32, ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    ref, ref_idx, rc = orc.decode_step(list(wl.modes), [W.u16(x[0]) for x in layers],
                                       [W.u16(x[1]) for x in layers],
                                       [W.u16(x[2]) for x in layers], lens, wl.top_k, shape.scale)
    assert rc == 0
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    for layer in range(wl.layers):
        check_outputs(outs[layer], outs32[layer], ref[layer], f"layer {layer}")


def test_plan_replays_the_step_bitwise():
    wl, layers = _tiny_inputs()
    shape = td.make_shape(wl.batch, wl.q_heads, wl.kv_heads, wl.max_seq_len)
    q = [x[0].cuda() for x in layers]
    K = [x[1].cuda() for x in layers]
    V = [x[2].cuda() for x in layers]
    seq = torch.as_tensor(W.seq_lens(wl)).cuda()
    res = []
    for use_plan in (False, True):
        outs = [torch.zeros_like(x) for x in q]
        outs32 = [torch.zeros(x.shape, dtype=torch.float32, device="cuda") for x in q]
        idx = torch.full((1, wl.kv_heads, wl.top_k), -1, dtype=torch.int32, device="cuda")
        ws = td.Workspace(shape, wl.top_k)
        if use_plan:
            plan = td.Plan(shape, wl.modes, q, K, V, seq, wl.top_k, idx, outs, outs32, ws)
            plan.launch()
            plan.launch()                   # replays leave the workspace reusable
            plan.close()
        else:
            td.td_decode_step(shape, wl.modes, q, K, V, seq, wl.top_k, idx, outs, outs32, ws)
        torch.cuda.synchronize()
        res.append((idx.clone(), [o.clone() for o in outs32]))
    assert torch.equal(res[0][0], res[1][0])
    for a, b in zip(res[0][1], res[1][1]):
        assert torch.equal(a, b)


def test_layer_events_time_each_layer():
    wl, layers = _tiny_inputs()
    shape = td.make_shape(wl.batch, wl.q_heads, wl.kv_heads, wl.max_seq_len)
    q = [x[0].cuda() for x in layers]
    K = [x[1].cuda() for x in layers]
    V = [x[2].cuda() for x in layers]
    outs = [torch.empty_like(x) for x in q]
    idx = torch.full((1, wl.kv_heads, wl.top_k), -1, dtype=torch.int32, device="cuda")
    ws = td.Workspace(shape, wl.top_k)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(wl.layers + 1)]
    td.td_decode_step(shape, wl.modes, q, K, V, torch.as_tensor(W.seq_lens(wl)).cuda(),
                      wl.top_k, idx, outs, None, ws, layer_events=ev)
    torch.cuda.synchronize()
    times = [ev[i].elapsed_time(ev[i + 1]) for i in range(wl.layers)]
    assert all(t > 0 for t in times)


def test_sparse_before_selection_launches_nothing():
    shape = td.make_shape(1, 2, 2, 64)
    x = torch.zeros(1, 2, D, dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros(1, 2, 64, D, dtype=torch.bfloat16, device="cuda")
    seq = torch.tensor([64], dtype=torch.int32, device="cuda")
    idx = torch.zeros(1, 2, 4, dtype=torch.int32, device="cuda")
    ws = td.Workspace(shape, 4)
    with pytest.raises(td.TdError) as e:
        td.td_decode_step(shape, [td.MODE_FULL, td.MODE_SPARSE], [x, x], [kv, kv], [kv, kv], seq,
                          4, idx, [x, x], None, ws)
    assert e.value.status == 3
    # with a caller-provided set the same schedule is accepted
    td.td_decode_step(shape, [td.MODE_FULL, td.MODE_SPARSE], [x, x], [kv, kv], [kv, kv], seq, 4,
                      idx, [x.clone(), x.clone()], None, ws, idx_valid=True)
    torch.cuda.synchronize()


@pytest.mark.parametrize("sparse", [False, True])
def test_cluster_and_global_split_merges_agree(orc, sparse):
    """The splits of a (batch, KV head) merge either through a thread-block
    cluster or through global partials and a ticket; both match the oracle."""
    G, Hkv, B, N = 4, 2, 3, 3000
    lens = [3000, 1111, 70]
    shape = td.make_shape(B, G * Hkv, Hkv, N, scale=td.default_scale(D))
    q, K, V, _ = W.random_case(50 + sparse, B, G * Hkv, Hkv, N, lens)
    idx = W.random_index_sets(52, B, Hkv, 900, lens, pad_fraction=0.05)
    res = {}
    try:
        for mode in (1, -1):
            td.td_set_tuning("cluster", mode)
            td.td_set_tuning("max_splits", 12)
            if sparse:
                out, out32, st = run_sparse(shape, q, K, V, lens, idx, 900)
                assert st == 0
            else:
                out, out32, _, _ = run_full(shape, q, K, V, lens)
            res[mode] = (out, out32)
    finally:
        td.td_set_tuning("cluster", 0)
        td.td_set_tuning("max_splits", 0)
    ref = oracle_sparse(orc, shape, q, K, V, idx) if sparse else oracle_full(orc, shape, q, K, V, lens)
    for mode, (out, out32) in res.items():
        check_outputs(out, out32, ref, f"merge mode {mode}")
    rowmax = res[-1][1].abs().amax(dim=-1, keepdim=True).clamp_min(1e-6)
    assert ((res[1][1] - res[-1][1]).abs() / rowmax).max().item() <= 2e-6


def _sorted_sets(rs, rows, k, n, short_every=3):
    out = np.full((rows, k), -1, np.int32)
    for r in range(rows):
        m = k if r % short_every else rs.randint(0, k + 1)       # some rows shorter than k
        out[r, :m] = np.sort(rs.choice(n, m, replace=False))
    return out


@pytest.mark.parametrize("k,n", [(1, 4), (7, 20), (512, 10240), (4096, 102400), (4096, 5000)])
def test_index_overlap_random_sets(orc, k, n):
    rs = np.random.RandomState(k + n)
    B, Hkv = 3, 4
    shape = td.make_shape(B, Hkv, Hkv, max(n, k))
    a = _sorted_sets(rs, B * Hkv, k, n)
    b = _sorted_sets(rs, B * Hkv, k, n)
    b[0] = a[0]                                                   # identical row
    counts = torch.full((B, Hkv), -5, dtype=torch.int32, device="cuda")
    td.td_index_overlap(shape, torch.as_tensor(a).cuda(), torch.as_tensor(b).cuda(), k, counts)
    got = counts.cpu().numpy().reshape(-1)
    want = [orc.index_overlap(a[r], b[r]) for r in range(B * Hkv)]
    assert got.tolist() == want


def test_index_overlap_of_consecutive_selection_layers(orc):
    """Figure 4(a)'s measure on a workload: the sets two selection layers pick
    (through the library) overlap exactly as the oracle counts them."""
    wl = W.WORKLOADS["llama2-7b-10k"].with_(max_seq_len=2048, top_k=128)
    lens = W.seq_lens(wl)
    heavy = W.heavy_positions(wl)
    shape = td.make_shape(wl.batch, wl.q_heads, wl.kv_heads, wl.max_seq_len,
                          scale=td.default_scale(D))
    seq = torch.as_tensor(lens).cuda()
    sets = []
    for layer in (1, 2):
        q, K, V = W.generate_layer(wl, layer, torch.device("cuda"), heavy[layer])
        idx = torch.full((wl.batch, wl.kv_heads, wl.top_k), -1, dtype=torch.int32, device="cuda")
        out = torch.empty_like(q)
        td.td_full_attn_select(shape, q, K, V, seq, wl.top_k, idx, out, None, None,
                               td.Workspace(shape, wl.top_k))
        sets.append(idx)
    counts = torch.empty((wl.batch, wl.kv_heads), dtype=torch.int32, device="cuda")
    td.td_index_overlap(shape, sets[0], sets[1], wl.top_k, counts)
    a, b = sets[0].cpu().numpy().reshape(-1, wl.top_k), sets[1].cpu().numpy().reshape(-1, wl.top_k)
    assert counts.cpu().numpy().reshape(-1).tolist() == [orc.index_overlap(a[r], b[r])
                                                        for r in range(len(a))]
    assert 0 <= counts.min().item() and counts.max().item() <= wl.top_k


def _coverage_ok(orc, s_ref, tau, k_max, k_got):
    """k_got is the oracle's budget, or one off where the cumulative mass at the
    cut is within fp32 rounding of 1 - tau (the kernel sums masses in fp32)."""
    k_ref = orc.coverage_count(s_ref, tau, k_max)
    if k_got == k_ref:
        return True
    if abs(k_got - k_ref) != 1:
        return False
    p = np.exp(s_ref - s_ref.max())
    p /= p.sum()
    order = np.lexsort((np.arange(len(s_ref)), -s_ref))
    cut = np.cumsum(p[order])[min(k_got, k_ref) - 1]
    return abs(cut - (1.0 - tau)) <= 1e-5


@pytest.mark.parametrize("G,tau,k_max,qscale", [(1, 0.1, 2000, 3.0), (1, 0.5, 64, 3.0),
                                                 (4, 0.01, 3000, 3.0), (2, 0.3, 1000, 3.0),
                                                 (8, 0.05, 500, 3.0), (1, 0.2, 300, 200.0)])
def test_coverage_selection(orc, G, tau, k_max, qscale):
    """qscale 200 gives scores in the hundreds: the kernel's histogram bound on
    the maximum is too coarse there and it takes the exact maximum instead."""
    Hkv, B, N = 2, 3, 3000
    lens = [3000, 1777, 40]
    shape = td.make_shape(B, G * Hkv, Hkv, N, scale=td.default_scale(D))
    q, K, V, _ = W.random_case(60 + G, B, G * Hkv, Hkv, N, lens)
    q = (q.float() * qscale).to(torch.bfloat16)   # peakier attention: budgets well below N
    qd, Kd, Vd = _dev(q, K, V)
    seq = torch.as_tensor(np.asarray(lens, np.int32)).cuda()
    idx = torch.full((B, Hkv, k_max), -7, dtype=torch.int32, device="cuda")
    counts = torch.full((B, Hkv), -7, dtype=torch.int32, device="cuda")
    out = torch.empty_like(qd)
    out32 = torch.empty(qd.shape, dtype=torch.float32, device="cuda")
    ws = td.Workspace(shape, k_max)
    td.td_full_attn_select_coverage(shape, qd, Kd, Vd, seq, tau, k_max, idx, counts, out, out32,
                                    None, ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    check_outputs(out, out32, oracle_full(orc, shape, q, K, V, lens), "coverage layer outputs")
    qb, Kb = W.u16(q), W.u16(K)
    idx, counts = idx.cpu().numpy(), counts.cpu().numpy()
    for b in range(B):
        for g in range(Hkv):
            s_ref = orc.group_scores(qb[b, g * G:(g + 1) * G], Kb[b, g], lens[b], shape.scale)
            k_got = int(counts[b, g])
            assert _coverage_ok(orc, s_ref, tau, k_max, k_got), f"b{b} g{g}: k={k_got}"
            assert np.all(idx[b, g, k_got:] == -1)
            ref_idx = orc.topk(s_ref, k_got)
            check_index_set(idx[b, g, :k_got], ref_idx, s_ref, k_got, f"b{b} g{g}")


@pytest.mark.parametrize("sparse", [False, True])
def test_probe_reads_exactly_the_layer_rows(sparse):
    """The read probe touches exactly the K/V rows its layer reads: the XOR of
    everything it folds equals the XOR of those rows' words."""
    G, Hkv, B, N, k = 2, 2, 3, 1500, 200
    lens = [1500, 777, 50]
    shape = td.make_shape(B, G * Hkv, Hkv, N)
    _, K, V, _ = W.random_case(70, B, G * Hkv, Hkv, N, lens)
    rs = np.random.RandomState(71)
    idx = np.full((B, Hkv, k), -1, np.int32)
    for b in range(B):
        for g in range(Hkv):
            m = min(k, lens[b])
            idx[b, g, :m] = np.sort(rs.choice(lens[b], m, replace=False))
    sink = torch.zeros(512, dtype=torch.int32, device="cuda")
    td.td_probe_layer_reads(shape, K.cuda(), V.cuda(), torch.tensor(lens, dtype=torch.int32).cuda(),
                            torch.as_tensor(idx).cuda() if sparse else None, k, sink)
    torch.cuda.synchronize()
    got = np.bitwise_xor.reduce(sink.cpu().numpy().view(np.uint32))
    kw = W.u16(K).view(np.uint32).reshape(B, Hkv, N, 64)
    vw = W.u16(V).view(np.uint32).reshape(B, Hkv, N, 64)
    want = np.uint32(0)
    for b in range(B):
        for g in range(Hkv):
            rows = idx[b, g][idx[b, g] >= 0] if sparse else np.arange(lens[b])
            want ^= np.bitwise_xor.reduce(kw[b, g, rows].ravel(), initial=np.uint32(0))
            want ^= np.bitwise_xor.reduce(vw[b, g, rows].ravel(), initial=np.uint32(0))
    assert got == want
