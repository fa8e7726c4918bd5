"""td_sparse_attn_noalloc: the sparse attention layer for callers that cannot
allocate device memory (no workspace; its scratch is a fixed array inside the
library).  It must give the same result as td_sparse_attn, the entry point
that uses a caller-provided workspace, on two calls in a row (the second call
finds the first call's leftovers in the shared scratch).

This file is collected last on purpose, and it also passes on its own in a
fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import sparse_attention_td_gb300 as td
import workloads as W
from parity_util import BF16_ATOL, F32_RTOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _case(seed, G, Hkv, B, N, lens, k, pad):
    shape = td.make_shape(B, G * Hkv, Hkv, N, scale=td.default_scale(128))
    q, K, V, _ = W.random_case(seed, B, G * Hkv, Hkv, N, lens)
    idx = W.random_index_sets(seed + 1, B, Hkv, k, lens, pad_fraction=pad)
    dev = [t.cuda() for t in (q, K, V)]
    seq = torch.as_tensor(np.asarray(lens, np.int32)).cuda()
    return shape, dev, seq, torch.as_tensor(idx).cuda()


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


def _same(a, b):
    (ob, of), (rb, rf) = a, b
    assert (ob.float() - rb.float()).abs().max().item() <= BF16_ATOL
    rowmax = rf.abs().amax(dim=-1, keepdim=True).clamp_min(1e-6)
    assert ((of - rf).abs() / rowmax).max().item() <= F32_RTOL


def test_no_alloc_matches_workspace_entry_point_on_two_calls():
    cases = [
        _case(70, 4, 2, 3, 3000, [3000, 1700, 640], 700, 0.1),   # several splits, padding
        _case(71, 1, 4, 2, 1024, [1024, 300], 64, 0.0),          # one split, different shape
    ]
    results = []
    for shape, (q, K, V), seq, idx in cases:
        k = idx.shape[-1]
        ref = _with_workspace(shape, q, K, V, seq, idx, k)
        got = _no_alloc_through_c_abi(shape, q, K, V, seq, idx, k)
        torch.cuda.synchronize()
        results.append((got, ref))
    for got, ref in results:
        _same(got, ref)


def test_no_alloc_rejects_what_the_fixed_scratch_cannot_hold():
    shape = td.make_shape(65535, 8, 8, 1 << 20)     # huge batch x heads: partials cannot fit
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    p = dummy.data_ptr()
    st = td.lib().td_sparse_attn_noalloc(ctypes.byref(shape), p, p, p, p, p, 1 << 17, p, None,
                                         None)
    assert st == 4   # TD_ERR_WORKSPACE_TOO_SMALL, nothing launched
