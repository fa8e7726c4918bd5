"""KV append through the C ABI against the definition: the new token's K/V rows
written at position seq_lens[b] - 1 of each layer's cache, then the step as
the oracle computes it on those caches.

The cache rows at the append positions start out as garbage, so a kernel that
read the stale row instead of the new one would fail the comparison."""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_td_gb300 as td
import workloads as W
from parity_util import check_outputs

pytestmark = pytest.mark.gpu
D = 128


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


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


@pytest.fixture(params=list(PATHS))
def staged(request):
    for key, value in PATHS[request.param].items():
        td.td_set_tuning(key, value)
    yield request.param
    for key in TUNING_KEYS:
        td.td_set_tuning(key, -1)


def _case(seed, B, Hq, Hkv, N, lens, layers, heavy_new=True):
    """Per-layer q, K, V with garbage at the append positions, and the new rows.
    heavy_new: the new key is aligned with its group's queries, so selection
    layers pick it and sparse layers must read it from the new rows."""
    g = torch.Generator().manual_seed(seed)
    G = Hq // Hkv
    out = []
    for _ in range(layers):
        q = torch.randn(B, Hq, D, generator=g).to(torch.bfloat16)
        K = torch.randn(B, Hkv, N, D, generator=g).to(torch.bfloat16)
        V = torch.randn(B, Hkv, N, D, generator=g).to(torch.bfloat16)
        k_new = torch.randn(B, Hkv, D, generator=g)
        if heavy_new:
            k_new += 0.5 * q.float().view(B, Hkv, G, D).sum(2)
        k_new = k_new.to(torch.bfloat16)
        v_new = torch.randn(B, Hkv, D, generator=g).to(torch.bfloat16)
        for b in range(B):
            if lens[b] > 0:      # stale contents the kernels must not use
                K[b, :, lens[b] - 1] = 30.0
                V[b, :, lens[b] - 1] = -30.0
        out.append((q, K, V, k_new, v_new))
    return out


def _appended(K, k_new, lens):
    K = K.clone()
    for b in range(K.shape[0]):
        if 1 <= lens[b] <= K.shape[2]:
            K[b, :, lens[b] - 1] = k_new[b]
    return K


def test_kv_append_writes_the_rows():
    B, Hkv, N = 3, 4, 300
    lens = [300, 17, 0]                    # a full row, a short one, nothing to append
    g = torch.Generator().manual_seed(3)
    K = torch.randn(B, Hkv, N, D, generator=g).to(torch.bfloat16)
    V = torch.randn(B, Hkv, N, D, generator=g).to(torch.bfloat16)
    kn = torch.randn(B, Hkv, D, generator=g).to(torch.bfloat16)
    vn = torch.randn(B, Hkv, D, generator=g).to(torch.bfloat16)
    shape = td.make_shape(B, Hkv, Hkv, N)
    Kd, Vd = K.cuda(), V.cuda()
    td.td_kv_append(shape, Kd, Vd, kn.cuda(), vn.cuda(), torch.tensor(lens, dtype=torch.int32).cuda())
    torch.cuda.synchronize()
    assert torch.equal(Kd.cpu(), _appended(K, kn, lens))
    assert torch.equal(Vd.cpu(), _appended(V, vn, lens))


@pytest.mark.parametrize("G", [1, 4])
@pytest.mark.parametrize("schedule", ["figure2", "per_layer_select"])
def test_append_step_matches_oracle(orc, staged, G, schedule):
    Hkv, B, N, k = 2, 2, 3000, 64
    Hq = G * Hkv
    lens = [3000, 1234]
    modes = (W.figure2_schedule(5, 3) if schedule == "figure2"
             else W.per_layer_select_schedule(5))
    layers = _case(40 + G, B, Hq, Hkv, N, lens, len(modes))
    shape = td.make_shape(B, Hq, Hkv, N, scale=td.default_scale(D))
    dev = [[t.cuda() for t in lay] for lay in layers]
    q = [x[0] for x in dev]
    K = [x[1] for x in dev]
    V = [x[2] for x in dev]
    kn = [x[3] for x in dev]
    vn = [x[4] for x in dev]
    outs = [torch.empty_like(x) for x in q]
    outs32 = [torch.empty(x.shape, dtype=torch.float32, device="cuda") for x in q]
    idx = torch.full((B, Hkv, k), -1, dtype=torch.int32, device="cuda")
    ws = td.Workspace(shape, k)
    seq = torch.tensor(lens, dtype=torch.int32).cuda()
    td.td_decode_step(shape, modes, q, K, V, seq, k, idx, outs, outs32, ws, k_new=kn, v_new=vn)
    torch.cuda.synchronize()
    assert ws.status() == 0
    Ka = [_appended(lay[1], lay[3], lens) for lay in layers]
    Va = [_appended(lay[2], lay[4], lens) for lay in layers]
    for layer in range(len(modes)):                       # the caches now hold the new rows
        assert torch.equal(K[layer].cpu(), Ka[layer])
        assert torch.equal(V[layer].cpu(), Va[layer])
    ref, ref_idx, rc = orc.decode_step(list(modes), [W.u16(lay[0]) for lay in layers],
                                       [W.u16(x) for x in Ka], [W.u16(x) for x in Va], lens, k,
                                       shape.scale)
    assert rc == 0
    got_idx = idx.cpu().numpy()
    assert np.array_equal(got_idx, ref_idx)
    for b in range(B):                                    # the new token was selected
        assert (got_idx[b] == lens[b] - 1).any(axis=-1).all()
    for layer in range(len(modes)):
        check_outputs(outs[layer], outs32[layer], ref[layer], f"layer {layer}")


def test_step_append_equals_append_then_step():
    """td_decode_step_append == td_kv_append on every layer + td_decode_step,
    bit for bit (same kernels, same split plan), also as a replayed plan."""
    Hkv, G, B, N, k = 4, 2, 2, 5000, 128
    lens = [5000, 2500]
    modes = W.figure2_schedule(6, 4)
    layers = _case(7, B, G * Hkv, Hkv, N, lens, len(modes))
    shape = td.make_shape(B, G * Hkv, Hkv, N, scale=td.default_scale(D))
    seq = torch.tensor(lens, dtype=torch.int32).cuda()

    def run(in_step, plan=False):
        dev = [[t.cuda() for t in lay] for lay in layers]
        q, K, V, kn, vn = ([x[i] for x in dev] for i in range(5))
        outs = [torch.empty_like(x) for x in q]
        idx = torch.full((B, Hkv, k), -1, dtype=torch.int32, device="cuda")
        ws = td.Workspace(shape, k)
        if in_step and plan:
            p = td.Plan(shape, modes, q, K, V, seq, k, idx, outs, None, ws, k_new=kn, v_new=vn)
            p.launch()
            p.launch()      # replaying rewrites the same rows: same result
        elif in_step:
            td.td_decode_step(shape, modes, q, K, V, seq, k, idx, outs, None, ws, k_new=kn,
                              v_new=vn)
        else:
            for layer in range(len(modes)):
                td.td_kv_append(shape, K[layer], V[layer], kn[layer], vn[layer], seq)
            td.td_decode_step(shape, modes, q, K, V, seq, k, idx, outs, None, ws)
        torch.cuda.synchronize()
        return [o.cpu() for o in outs], idx.cpu(), [x.cpu() for x in K + V]

    base = run(False)
    for variant in (run(True), run(True, plan=True)):
        assert all(torch.equal(a, b) for a, b in zip(base[0], variant[0]))
        assert torch.equal(base[1], variant[1])
        assert all(torch.equal(a, b) for a, b in zip(base[2], variant[2]))


def test_growing_context_over_steps(orc):
    """Three decode steps, each appending one token (seq_lens + 1 per step),
    against the oracle on the grown caches."""
    Hkv, G, B, N, k = 2, 4, 1, 1024, 32
    modes = W.figure2_schedule(5, 3)          # full, full, select, select, sparse
    shape = td.make_shape(B, G * Hkv, Hkv, N, scale=td.default_scale(D))
    layers = _case(9, B, G * Hkv, Hkv, N, [N], len(modes), heavy_new=False)
    Kc = [lay[1].clone() for lay in layers]
    Vc = [lay[2].clone() for lay in layers]
    K = [x.cuda() for x in Kc]
    V = [x.cuda() for x in Vc]
    q = [lay[0].cuda() for lay in layers]
    outs = [torch.empty_like(x) for x in q]
    outs32 = [torch.empty(x.shape, dtype=torch.float32, device="cuda") for x in q]
    idx = torch.full((B, Hkv, k), -1, dtype=torch.int32, device="cuda")
    ws = td.Workspace(shape, k)
    g = torch.Generator().manual_seed(10)
    for n in (600, 601, 602):
        lens = [n]
        kn = [torch.randn(B, Hkv, D, generator=g).to(torch.bfloat16) for _ in modes]
        vn = [torch.randn(B, Hkv, D, generator=g).to(torch.bfloat16) for _ in modes]
        td.td_decode_step(shape, modes, q, K, V, torch.tensor(lens, dtype=torch.int32).cuda(), k,
                          idx, outs, outs32, ws, k_new=[x.cuda() for x in kn],
                          v_new=[x.cuda() for x in vn])
        torch.cuda.synchronize()
        Kc = [_appended(Kc[layer], kn[layer], lens) for layer in range(len(modes))]
        Vc = [_appended(Vc[layer], vn[layer], lens) for layer in range(len(modes))]
        ref, ref_idx, rc = orc.decode_step(list(modes), [W.u16(x) for x in q],
                                           [W.u16(x) for x in Kc], [W.u16(x) for x in Vc], lens,
                                           k, shape.scale)
        assert rc == 0
        assert np.array_equal(idx.cpu().numpy(), ref_idx)
        for layer in range(len(modes)):
            check_outputs(outs[layer], outs32[layer], ref[layer], f"n={n} layer {layer}")


def test_append_over_more_layers_than_one_launch_takes(orc):
    """40 layers: the step appends in two launches (32 + 8 layers); every
    layer's cache gets its row and every layer attends to it."""
    L, Hkv, G, B, N = 40, 2, 1, 2, 160
    lens = [160, 77]
    modes = [W.FULL] * L
    layers = _case(21, B, G * Hkv, Hkv, N, lens, L, heavy_new=False)
    shape = td.make_shape(B, G * Hkv, Hkv, N, scale=td.default_scale(D))
    dev = [[t.cuda() for t in lay] for lay in layers]
    q, K, V, kn, vn = ([x[i] for x in dev] for i in range(5))
    outs = [torch.empty_like(x) for x in q]
    outs32 = [torch.empty(x.shape, dtype=torch.float32, device="cuda") for x in q]
    ws = td.Workspace(shape, 0)
    td.td_decode_step(shape, modes, q, K, V, torch.tensor(lens, dtype=torch.int32).cuda(), 0, None,
                      outs, outs32, ws, k_new=kn, v_new=vn)
    torch.cuda.synchronize()
    for layer in range(L):
        Ka = _appended(layers[layer][1], layers[layer][3], lens)
        Va = _appended(layers[layer][2], layers[layer][4], lens)
        assert torch.equal(K[layer].cpu(), Ka) and torch.equal(V[layer].cpu(), Va), layer
        if layer in (0, 31, 32, 39):
            qb, Kb, Vb = W.u16(layers[layer][0]), W.u16(Ka), W.u16(Va)
            ref = np.zeros((B, G * Hkv, D))
            for b in range(B):
                for h in range(G * Hkv):
                    ref[b, h] = orc.attend(qb[b, h], Kb[b, h // G, :lens[b]], Vb[b, h // G, :lens[b]],
                                           shape.scale)
            check_outputs(outs[layer], outs32[layer], ref, f"layer {layer}")
