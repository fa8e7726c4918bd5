"""Comparison rules between the CUDA path and the oracle.

Outputs: the bf16 output within max-abs 2e-2 of the fp64 oracle; the fp32
output per (batch, head) row within 1e-5 x max(max |oracle row|, 1e-6).
Index sets: equal, or differing only by swaps among positions whose oracle
scores lie within 1e-3 x |s_k| of the k-th largest oracle score s_k (the tie
rule for fp32-vs-fp64 selection scores).  Positions whose scores equal s_k
exactly (the tie itself) always pass.
"""
from __future__ import annotations

import numpy as np
import torch

BF16_ATOL = 2e-2
F32_RTOL = 1e-5
SET_RTOL = 1e-3


def check_outputs(out_bf16: torch.Tensor, out_f32: torch.Tensor, ref: np.ndarray, what=""):
    """out_*: [..., d] tensors; ref: float64 array of the same shape."""
    ob = out_bf16.float().cpu().double().numpy().reshape(ref.shape)
    of = out_f32.cpu().double().numpy().reshape(ref.shape)
    err_b = np.max(np.abs(ob - ref)) if ref.size else 0.0
    assert err_b <= BF16_ATOL, f"{what}: bf16 max-abs {err_b:.3e} > {BF16_ATOL}"
    rowmax = np.maximum(np.abs(ref).max(axis=-1, keepdims=True), 1e-6)
    rel = np.abs(of - ref) / rowmax
    worst = float(rel.max()) if rel.size else 0.0
    assert worst <= F32_RTOL, f"{what}: fp32 row-relative error {worst:.3e} > {F32_RTOL}"
    return err_b, worst


def check_index_set(got: np.ndarray, ref: np.ndarray, s_ref: np.ndarray, k: int, what="") -> bool:
    """True if identical; False if they differ only by tolerated swaps
    (asserts otherwise)."""
    got = np.asarray(got)
    ref = np.asarray(ref)
    g_live = got[got >= 0]
    r_live = ref[ref >= 0]
    assert np.all(np.diff(g_live) > 0), f"{what}: indices not ascending/distinct"
    assert np.all(got[len(g_live):] == -1), f"{what}: padding not at the end"
    assert len(g_live) == len(r_live), f"{what}: {len(g_live)} vs {len(r_live)} positions"
    if np.array_equal(g_live, r_live):
        return True
    n = len(s_ref)
    assert g_live.max() < n, f"{what}: index out of range"
    kth = np.sort(s_ref)[::-1][min(k, n) - 1]
    tol = SET_RTOL * abs(kth)
    diff = np.setxor1d(g_live, r_live)
    bad = diff[np.abs(s_ref[diff] - kth) > tol]
    assert bad.size == 0, (f"{what}: positions {bad[:8]} differ with scores "
                           f"{s_ref[bad[:8]]} vs k-th {kth}")
    return False
