"""The C-ABI library on the host: it loads, exports every declared symbol,
sizes workspaces without a GPU, and rejects bad arguments before launching
anything (so none of these calls touches device memory)."""
import ctypes
import os
import re

import pytest

import sparse_attention_td_gb300 as td
from sparse_attention_td_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "td.h")

INVALID, UNSUPPORTED, NO_SEL, WS_SMALL = 1, 2, 3, 4


@pytest.fixture(scope="module")
def L():
    libbuild.build()
    return td.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(td_[a-z_]+)\s*\(", text)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(L, n), f"{n} declared in td.h but not exported"


def test_status_strings(L):
    for code, name in [(0, "TD_OK"), (1, "TD_ERR_INVALID_ARG"), (3, "TD_ERR_NO_SELECTION"),
                       (5, "TD_ERR_CUDA")]:
        assert td.td_status_string(code) == name


def shape(**kw):
    base = dict(batch=2, num_q_heads=8, num_kv_heads=2, max_seq_len=1000, head_dim=128, scale=0.0)
    base.update(kw)
    return td.Shape(base["batch"], base["num_q_heads"], base["num_kv_heads"], base["head_dim"],
                    base["max_seq_len"], base["scale"])


def test_workspace_size_is_host_only_and_monotone(L):
    s = shape()
    a = td.td_workspace_size(s, 0)
    b = td.td_workspace_size(s, 64)
    assert 0 < a < b
    assert b - a >= 2 * 2 * 1000 * 4        # the selection scores [B][Hkv][N] fp32
    assert td.td_workspace_size(shape(head_dim=64), 0) == 0
    assert td.td_workspace_size(shape(num_q_heads=12, num_kv_heads=4), 0) == 0   # G = 3
    assert td.td_workspace_size(s, 1001) == 0                                     # k > N


def test_default_scale_is_fp32_inverse_sqrt():
    import numpy as np
    assert td.default_scale(128) == float(np.float32(1) / np.sqrt(np.float32(128)))


FAKE = 1 << 20   # aligned but never dereferenced: every call below fails validation first


def _full(L, s, q=FAKE, k=FAKE, v=FAKE, seq=FAKE, top_k=0, idx=None, out=FAKE, ws=FAKE,
          ws_bytes=None):
    if ws_bytes is None:
        ws_bytes = 0
    return L.td_full_attn_select(ctypes.byref(s), q, k, v, seq, top_k, idx, out, None, None,
                                 ws, ws_bytes, None)


def test_full_rejects_bad_arguments(L):
    s = shape()
    need = td.td_workspace_size(s, 0)
    assert _full(L, None if False else s, q=None, ws_bytes=need) == INVALID
    assert _full(L, s, q=FAKE + 2, ws_bytes=need) == INVALID            # misaligned q
    assert _full(L, shape(head_dim=64), ws_bytes=need) == UNSUPPORTED
    assert _full(L, shape(num_q_heads=6, num_kv_heads=2), ws_bytes=need) == UNSUPPORTED
    assert _full(L, shape(num_q_heads=7, num_kv_heads=2), ws_bytes=need) == INVALID
    assert _full(L, s, ws_bytes=need - 1) == WS_SMALL
    assert _full(L, s, top_k=2000, ws_bytes=1 << 40) == INVALID         # k > N_max
    assert _full(L, s, top_k=8, idx=None, ws_bytes=1 << 40) == INVALID  # select needs idx
    assert _full(L, s, ws=FAKE + 16, ws_bytes=1 << 40) == INVALID       # ws alignment
    assert L.td_full_attn_select(None, FAKE, FAKE, FAKE, FAKE, 0, None, FAKE, None, None,
                                 FAKE, 1 << 40, None) == INVALID


def test_sparse_and_topk_reject_bad_arguments(L):
    s = shape()
    big = 1 << 40
    assert L.td_sparse_attn(ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, None, 8, FAKE, None,
                            FAKE, big, None) == INVALID                  # no idx
    assert L.td_sparse_attn(ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, FAKE, 0, FAKE, None,
                            FAKE, big, None) == INVALID                  # k = 0
    assert L.td_topk_select(ctypes.byref(s), None, FAKE, 8, FAKE, FAKE, big, None) == INVALID
    assert L.td_topk_select(ctypes.byref(s), FAKE, FAKE, 0, FAKE, FAKE, big, None) == INVALID


def _step(L, s, modes, idx_valid=0, top_k=8, idx=FAKE, ws_bytes=1 << 40):
    n = len(modes)
    arr = (ctypes.c_void_p * n)(*([FAKE] * n))
    m = (ctypes.c_int32 * n)(*modes)
    return L.td_decode_step(ctypes.byref(s), n, m, arr, arr, arr, FAKE, top_k, idx, idx_valid,
                            arr, None, FAKE, ws_bytes, None, None)


def test_step_schedule_checks(L):
    s = shape()
    assert _step(L, s, [0, 2]) == NO_SEL                 # sparse before any selection
    assert _step(L, s, [2, 1, 2]) == NO_SEL
    assert _step(L, s, [0, 7]) == INVALID                # unknown mode
    assert _step(L, s, [1, 2], top_k=0) == INVALID       # selection needs k >= 1
    assert _step(L, s, [1, 2], idx=None) == INVALID      # selection needs idx_buf
    assert _step(L, s, [0, 1, 2], ws_bytes=16) == WS_SMALL


def test_tuning_keys(L):
    td.td_set_tuning("full_waves", 3)
    td.td_set_tuning("full_waves", 0)     # default again
    td.td_set_tuning("topk_threads", 512)
    td.td_set_tuning("topk_threads", 0)
    td.td_set_tuning("pdl", 0)
    td.td_set_tuning("pdl", 1)
    td.td_set_tuning("mma", 0)
    td.td_set_tuning("mma", -1)
    td.td_set_tuning("full_prefetch", 2)
    td.td_set_tuning("full_prefetch", -1)
    td.td_set_tuning("topk_warp_max", 2048)
    td.td_set_tuning("topk_warp_max", 0)
    for key, value in (("mma_full_tokens", 8), ("mma_sparse_tokens", 32), ("mma_sparse_tokens", 64),
                       ("topk_cluster", 4), ("sparse_staged", 2), ("full_interleave", 0),
                       ("early_trigger", 0), ("sparse_splits", 5), ("host_copy", 0),
                       ("wait_limit_us", 50), ("wait_test", 1)):
        td.td_set_tuning(key, value)
        td.td_set_tuning(key, -1 if key not in ("wait_limit_us", "wait_test") else 0)
    with pytest.raises(td.TdError):
        td.td_set_tuning("no_such_knob", 1)


def test_kernel_name_of_an_invalid_shape(L):
    assert td.td_kernel_name(shape(head_dim=64), 0, False) == "invalid shape"
    assert td.td_kernel_name(shape(), -1, True) == "invalid shape"


def test_index_overlap_rejects_bad_arguments(L):
    s = shape()
    p = ctypes.c_void_p(256)     # never dereferenced: validation fails first
    assert L.td_index_overlap(ctypes.byref(s), None, p, 8, p, None) == INVALID
    assert L.td_index_overlap(ctypes.byref(s), p, None, 8, p, None) == INVALID
    assert L.td_index_overlap(ctypes.byref(s), p, p, 8, None, None) == INVALID
    assert L.td_index_overlap(ctypes.byref(s), p, p, 0, p, None) == INVALID
    assert L.td_index_overlap(ctypes.byref(s), ctypes.c_void_p(258), p, 8, p, None) == INVALID
    assert L.td_index_overlap(ctypes.byref(shape(head_dim=64)), p, p, 8, p, None) == UNSUPPORTED


def test_probe_rejects_bad_arguments(L):
    s = shape()
    p = ctypes.c_void_p(256)
    assert L.td_probe_layer_reads(ctypes.byref(s), None, p, p, None, 0, p, 4, None) == INVALID
    assert L.td_probe_layer_reads(ctypes.byref(s), p, p, p, None, 0, p, 0, None) == INVALID
    assert L.td_probe_layer_reads(ctypes.byref(s), p, p, p, p, 0, p, 4, None) == INVALID     # k < 1
    assert L.td_probe_layer_reads(ctypes.byref(s), p, p, p, p, 5000, p, 4, None) == INVALID  # k > N
