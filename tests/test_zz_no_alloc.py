"""td_sparse_attn_noalloc: the sparse attention layer for callers that cannot
allocate device memory (no workspace; its scratch is a fixed array inside the
library).  Its results must match the CPU oracle, and agree with
td_sparse_attn (the entry point that uses a caller-provided workspace) within
the parity tolerance, on calls in a row: every call after the first finds the
previous call's leftovers in the shared scratch.

This file is collected last on purpose, and it also passes on its own in a
fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import sparse_attention_td_gb300 as td
import workloads as W
from parity_util import BF16_ATOL, F32_RTOL, check_outputs

pytestmark = pytest.mark.gpu
D = 128


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _case(seed, G, Hkv, B, N, lens, k, pad):
    shape = td.make_shape(B, G * Hkv, Hkv, N, scale=td.default_scale(D))
    q, K, V, _ = W.random_case(seed, B, G * Hkv, Hkv, N, lens)
    idx = W.random_index_sets(seed + 1, B, Hkv, k, lens, pad_fraction=pad)
    return shape, (q, K, V), lens, idx


def _device(q, K, V, lens, idx):
    seq = torch.as_tensor(np.asarray(lens, np.int32)).cuda()
    return [t.cuda() for t in (q, K, V)], seq, torch.as_tensor(idx).cuda()


def _with_workspace(shape, q, K, V, seq, idx, k):
    out = torch.empty_like(q)
    out32 = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    ws = td.Workspace(shape, k)
    td.td_sparse_attn(shape, q, K, V, seq, idx, k, out, out32, ws)
    return out, out32


def _no_alloc_through_c_abi(shape, q, K, V, seq, idx, k):
    out = torch.empty_like(q)
    out32 = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    st = td.lib().td_sparse_attn_noalloc(
        ctypes.byref(shape), q.data_ptr(), K.data_ptr(), V.data_ptr(), seq.data_ptr(),
        idx.data_ptr(), k, out.data_ptr(), out32.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert st == 0, td.td_status_string(st)
    return out, out32


def _oracle(shape, q, K, V, lens, idx, rows=None):
    """fp64 oracle output [B][Hq][D] over each head's persisted positions
    (padding skipped); rows: optional list of (b, h) to compute (others 0)."""
    orc = oracle.get()
    G = shape.num_q_heads // shape.num_kv_heads
    qb, Kb, Vb = W.u16(q), W.u16(K), W.u16(V)
    ref = np.zeros((shape.batch, shape.num_q_heads, D))
    todo = rows if rows is not None else [(b, h) for b in range(shape.batch)
                                         for h in range(shape.num_q_heads)]
    for b, h in todo:
        g = h // G
        sel = idx[b, g]
        sel = sel[sel >= 0]
        ref[b, h] = orc.attend(qb[b, h], Kb[b, g, :lens[b]], Vb[b, g, :lens[b]], shape.scale,
                               rows=sel)
    return ref


def _agree(a, b):
    (ob, of), (rb, rf) = a, b
    assert (ob.float() - rb.float()).abs().max().item() <= BF16_ATOL
    rowmax = rf.abs().amax(dim=-1, keepdim=True).clamp_min(1e-6)
    assert ((of - rf).abs() / rowmax).max().item() <= F32_RTOL


def test_no_alloc_matches_the_oracle_and_the_workspace_entry_point_on_calls_in_a_row():
    cases = [
        _case(70, 4, 2, 3, 3000, [3000, 1700, 640], 700, 0.1),   # several splits, padding
        _case(71, 1, 4, 2, 1024, [1024, 300], 64, 0.0),          # one split, MHA
        _case(72, 8, 1, 2, 5000, [5000, 4100], 2500, 0.05),      # G = 8, many splits
        _case(70, 4, 2, 3, 3000, [3000, 1700, 640], 700, 0.1),   # the first case again
    ]
    for shape, host, lens, idx in cases:
        (q, K, V), seq, idxd = _device(*host, lens, idx)
        k = idx.shape[-1]
        got = _no_alloc_through_c_abi(shape, q, K, V, seq, idxd, k)
        ref_ws = _with_workspace(shape, q, K, V, seq, idxd, k)
        torch.cuda.synchronize()
        check_outputs(got[0], got[1], _oracle(shape, *host, lens, idx),
                      f"no-alloc G={shape.num_q_heads // shape.num_kv_heads} k={k}")
        _agree(got, ref_ws)


def test_no_alloc_takes_one_split_shapes_without_room_for_partials():
    """B * Hkv * G * (128 + 2) * 4 bytes of partials would exceed the scratch, but
    top_k fits one CTA: the call needs only tickets and is accepted."""
    B, Hkv, G, N, k = 64, 32, 8, 96, 64
    shape, host, lens, idx = _case(73, G, Hkv, B, N, [N - (b % 7) for b in range(B)], k, 0.1)
    assert B * Hkv * G * (D + 2) * 4 > td.NOALLOC_SCRATCH_BYTES
    (q, K, V), seq, idxd = _device(*host, lens, idx)
    for _ in range(2):
        got = _no_alloc_through_c_abi(shape, q, K, V, seq, idxd, k)
        torch.cuda.synchronize()
        rows = [(b, h) for b in (0, 13, 63) for h in (0, 77, 255)]
        ref = _oracle(shape, *host, lens, idx, rows)
        bs, hs = [r[0] for r in rows], [r[1] for r in rows]
        check_outputs(got[0][bs, hs], got[1][bs, hs], ref[bs, hs], "one-split no-alloc")


def test_no_alloc_rejects_what_the_fixed_scratch_cannot_hold():
    shape = td.make_shape(65535, 8, 8, 1 << 20)     # huge batch x heads: partials cannot fit
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    p = dummy.data_ptr()
    st = td.lib().td_sparse_attn_noalloc(ctypes.byref(shape), p, p, p, p, p, 1 << 17, p, None,
                                         None)
    assert st == 4   # TD_ERR_WORKSPACE_TOO_SMALL, nothing launched
