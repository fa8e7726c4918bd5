"""td_plan_create_host: a captured step that also copies every layer's q
rows in from page-locked host memory and the outputs back (one buffer per
side).  The device results must equal those of the plain plan bitwise,
launch after launch, and the host buffer must hold exactly the device
outputs once the stream is done -- with the copy kernels (the default) and
with the copy engines, on steps whose q rows exceed 1 MiB (the rows of
layers 1 .. L-1 come in beside layer 0) and whose outputs take several
side-stream copies.  Pageable host memory is rejected by the C call itself."""
import ctypes

import numpy as np
import pytest
import torch

import sparse_attention_td_gb300 as td
import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _workload(name, n_layers=4):
    wl = W.WORKLOADS[name]
    if name == "tiny" and n_layers < 4:   # one full+select layer, then at most one sparse layer
        wl = wl.with_(layers=n_layers, modes=(W.FULL_SELECT, W.SPARSE)[:n_layers])
    elif name != "tiny":   # a grouped-query workload, cut to a few layers of short rows
        modes = (W.FULL, W.FULL, W.FULL_SELECT) + (W.SPARSE,) * (n_layers - 3)
        if name == "serving-b32":
            wl = wl.with_(layers=n_layers, modes=modes, max_seq_len=1024, top_k=256,
                          ragged=(600, 1024))
        else:
            wl = wl.with_(layers=n_layers, modes=modes, max_seq_len=4096, top_k=512)
    heavy = W.heavy_positions(wl)
    layers = [W.generate_layer(wl, layer, "cpu", heavy[layer]) for layer in range(wl.layers)]
    return wl, layers


def _device_plan_run(wl, shape, q_rows, K, V, seq):
    q = [x.cuda() for x in q_rows]
    outs = [torch.zeros_like(x) for x in q]
    idx = torch.full((wl.batch, wl.kv_heads, wl.top_k), -1, dtype=torch.int32, device="cuda")
    ws = td.Workspace(shape, wl.top_k)
    plan = td.Plan(shape, wl.modes, q, K, V, seq, wl.top_k, idx, outs, None, ws)
    plan.launch()
    torch.cuda.synchronize()
    plan.close()
    return [o.cpu() for o in outs], idx.cpu()


# (workload, layers): 12 layers of the 32K shape take output copies of
# layers 0-7 and 8-9 on the side stream; 6 layers of the serving batch hold
# 1.5 MiB of q rows; one and two layers leave the side stream unused
CASES = [("tiny", 4), ("tiny", 1), ("tiny", 2), ("llama3-8b-32k", 12), ("serving-b32", 6)]


@pytest.mark.parametrize("host_copy", [1, 0], ids=["kernels", "engines"])
@pytest.mark.parametrize("name,n_layers", CASES, ids=[f"{c[0]}-L{c[1]}" for c in CASES])
def test_host_plan_equals_the_device_plan_on_every_launch(name, n_layers, host_copy):
    wl, layers = _workload(name, n_layers)
    shape = td.make_shape(wl.batch, wl.q_heads, wl.kv_heads, wl.max_seq_len)
    K = [x[1].cuda() for x in layers]
    V = [x[2].cuda() for x in layers]
    seq = torch.as_tensor(W.seq_lens(wl)).cuda()
    rows_shape = (wl.layers,) + tuple(layers[0][0].shape)
    q_all = torch.zeros(rows_shape, dtype=torch.bfloat16, device="cuda")
    outs_all = torch.zeros_like(q_all)
    q_host = torch.stack([x[0] for x in layers]).pin_memory()
    out_host = torch.full(rows_shape, float("nan"), dtype=torch.bfloat16).pin_memory()
    idx = torch.full((wl.batch, wl.kv_heads, wl.top_k), -1, dtype=torch.int32, device="cuda")
    ws = td.Workspace(shape, wl.top_k)
    td.td_set_tuning("host_copy", host_copy)
    try:
        plan = td.Plan(shape, wl.modes, list(q_all.unbind(0)), K, V, seq, wl.top_k, idx,
                       list(outs_all.unbind(0)), None, ws, q_host=q_host, out_host=out_host)
    finally:
        td.td_set_tuning("host_copy", -1)
    rs = np.random.RandomState(5)
    for launch in range(3):
        if launch > 0:   # new host q rows for this launch
            q_host.copy_(torch.as_tensor(rs.standard_normal(rows_shape).astype(np.float32))
                         .to(torch.bfloat16))
        rows = list(q_host.clone().unbind(0))
        plan.launch()
        torch.cuda.synchronize()
        ref_outs, ref_idx = _device_plan_run(wl, shape, rows, K, V, seq)
        assert torch.equal(idx.cpu(), ref_idx)
        assert torch.equal(q_all.cpu(), q_host)
        for layer in range(wl.layers):
            assert torch.equal(outs_all[layer].cpu(), ref_outs[layer])
            assert torch.equal(out_host[layer], ref_outs[layer])
    plan.close()
    assert ws.status() == 0


def test_pageable_or_scattered_buffers_are_rejected():
    wl, layers = _workload("tiny")
    shape = td.make_shape(wl.batch, wl.q_heads, wl.kv_heads, wl.max_seq_len)
    K = [x[1].cuda() for x in layers]
    V = [x[2].cuda() for x in layers]
    seq = torch.as_tensor(W.seq_lens(wl)).cuda()
    q_all = torch.stack([x[0] for x in layers]).cuda()
    outs_all = torch.zeros_like(q_all)
    idx = torch.full((wl.batch, wl.kv_heads, wl.top_k), -1, dtype=torch.int32, device="cuda")
    ws = td.Workspace(shape, wl.top_k)
    pinned = q_all.cpu().pin_memory()
    pinned_out = torch.empty_like(pinned).pin_memory()
    pageable = q_all.cpu()
    L = wl.layers
    arr = lambda ts: (ctypes.c_void_p * L)(*[t.data_ptr() for t in ts])
    modes = (ctypes.c_int32 * L)(*wl.modes)
    plan = ctypes.c_void_p(0)
    for q_host, out_host in ((pageable, pinned_out), (pinned, pageable)):
        st = td.lib().td_plan_create_host(
            ctypes.byref(plan), ctypes.byref(shape), L, modes, q_host.data_ptr(),
            q_all.data_ptr(), arr(K), arr(V), seq.data_ptr(), wl.top_k, idx.data_ptr(), 0,
            outs_all.data_ptr(), None, out_host.data_ptr(), ws.ptr, ws.nbytes)
        assert st == 1 and not plan.value   # TD_ERR_INVALID_ARG, no plan
    with pytest.raises(ValueError, match="page-locked"):
        td.Plan(shape, wl.modes, list(q_all.unbind(0)), K, V, seq, wl.top_k, idx,
                list(outs_all.unbind(0)), None, ws, q_host=pageable, out_host=pinned_out)
    gapped = torch.zeros((L, 2) + tuple(q_all.shape[1:]), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError, match="one bf16 buffer"):   # layers not back to back
        td.Plan(shape, wl.modes, list(gapped[:, 0].unbind(0)), K, V, seq, wl.top_k, idx,
                list(outs_all.unbind(0)), None, ws, q_host=pinned, out_host=pinned_out)
