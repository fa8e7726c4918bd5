"""Failure report of the staged full-layer kernel's bounded waits.

The staged kernel waits on an mbarrier for each stage of bulk copies, with a
time limit.  The test switch "wait_test" makes the first wait of every CTA
poll a barrier that nothing arrives on (a flag nobody sets), so every wait
runs out after "wait_limit_us": no fault, no hang.  Each CTA then waits for
the copies it issued, joins the split merge with an empty partial and sets
TD_FLAG_WAIT_TIMEOUT.  The checks:
  * the status word reports the timeout and the call returns normally;
  * every output is zero (every split gave up, so every merge saw only empty
    partials);
  * the next call on the same workspace, with the switch off, matches the
    oracle: the merge tickets returned to zero, so no stale partial is used.
"""
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
    yield
    for key in ("wait_test", "wait_limit_us", "full_staged", "mma", "max_splits"):
        td.td_set_tuning(key, -1 if key in ("full_staged", "mma") else 0)


@pytest.mark.parametrize("G,max_splits", [(4, 0), (4, 1), (1, 0)])
def test_staged_wait_runs_out_then_the_workspace_is_clean(G, max_splits):
    td.td_set_tuning("mma", 0)            # CUDA-core kernels
    td.td_set_tuning("full_staged", 1)    # K/V through the bulk-copy ring
    td.td_set_tuning("max_splits", max_splits)
    Hkv, B, N = 2, 3, 2000
    lens = [2000, 1333, 70]
    shape = td.make_shape(B, G * Hkv, Hkv, N, scale=td.default_scale(D))
    q, K, V, _ = W.random_case(90 + G, B, G * Hkv, Hkv, N, lens)
    qd, Kd, Vd = (t.cuda() for t in (q, K, V))
    seq = torch.as_tensor(np.asarray(lens, np.int32)).cuda()
    out = torch.full_like(qd, 1.0)
    out32 = torch.full(qd.shape, 1.0, dtype=torch.float32, device="cuda")
    ws = td.Workspace(shape, 0)

    td.td_set_tuning("wait_limit_us", 20)
    td.td_set_tuning("wait_test", 1)
    try:
        td.td_full_attn_select(shape, qd, Kd, Vd, seq, 0, None, out, out32, None, ws)
        torch.cuda.synchronize()
    finally:
        td.td_set_tuning("wait_test", 0)
        td.td_set_tuning("wait_limit_us", 0)
    assert ws.status() & td.FLAG_WAIT_TIMEOUT
    assert torch.all(out == 0) and torch.all(out32 == 0)

    td.td_full_attn_select(shape, qd, Kd, Vd, seq, 0, None, out, out32, None, ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    orc = oracle.get()
    qb, Kb, Vb = W.u16(q), W.u16(K), W.u16(V)
    ref = np.zeros((B, G * Hkv, D))
    for b in range(B):
        for h in range(G * Hkv):
            ref[b, h] = orc.attend(qb[b, h], Kb[b, h // G, :lens[b]], Vb[b, h // G, :lens[b]],
                                   shape.scale)
    check_outputs(out, out32, ref, f"after the timeout, G={G}")
    td.td_set_tuning("max_splits", 0)
