"""Seeded synthetic decode-step workloads (shared by the tests, the bench and smoke).

This module holds no attention arithmetic: it only draws inputs.  Both the
CUDA path and the CPU oracle consume the same generated bf16 tensors, so the
two sides never depend on each other.

The shapes follow the TidalDecode paper review page: LLaMA-2-7B and
LLaMA-3-8B attention shapes (§五 efficiency evaluation, 10K-100K contexts;
§五 table of optimal re-selection layers, L7 for LLaMA-2 and L14 for
LLaMA-3) and the per-step schedule of §三 Figure 2.  The pages evaluate on
real models and datasets; here K, V and q are i.i.d. N(0, 1) with a planted
set of "heavy" positions whose keys lean towards the queries, so that the
selected top-k sets are coherent across layers the way the review's
Figure 1 describes.  The recipe per workload is in ``WORKLOADS`` below.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np
import torch

FULL = 0
FULL_SELECT = 1
SPARSE = 2
MODE_NAMES = {FULL: "full", FULL_SELECT: "full+select", SPARSE: "sparse"}


def figure2_schedule(num_layers: int, middle: int) -> tuple[int, ...]:
    """Layer modes of one decode step (TidalDecode review §三 Figure 2).

    Layers 0 and 1 run full attention without selection, layer 2 runs full
    attention with token selection, layers 3..middle-1 are sparse (PPSA),
    layer ``middle`` selects again, and every later layer is sparse.
    """
    if num_layers < 3 or not (2 < middle < num_layers):
        raise ValueError("Figure 2 needs >= 3 layers and 2 < middle < num_layers")
    modes = []
    for layer in range(num_layers):
        if layer < 2:
            modes.append(FULL)
        elif layer == 2 or layer == middle:
            modes.append(FULL_SELECT)
        else:
            modes.append(SPARSE)
    return tuple(modes)


def all_full_schedule(num_layers: int) -> tuple[int, ...]:
    return tuple([FULL] * num_layers)


def per_layer_select_schedule(num_layers: int) -> tuple[int, ...]:
    """Token selection at every layer after the first two: the schedule whose
    selection cost the review compares PPSA against (per-layer selection as in
    Quest, §三 complexity comparison: L selections per step instead of 2).
    With these kernels every such layer pays full attention plus the top-k."""
    return tuple([FULL] * min(2, num_layers) + [FULL_SELECT] * max(0, num_layers - 2))


# Optimal re-selection ("middle") layer per model family, TidalDecode review
# §五 table: LLaMA-2-7B (LongChat, Yarn) -> L7, LLaMA-3-8B / 3.1-8B -> L14.
RESELECTION_LAYER = {"llama-2-7b": 7, "llama-3-8b": 14}


def kv_cache_bytes(layers: int, kv_heads: int, head_dim: int, tokens: int,
                   bytes_per_elem: int = 2) -> int:
    """KV-cache size: layers x KV heads x head_dim x tokens x bytes x 2 (K and V)
    (TidalDecode review §二 problem definition)."""
    return layers * kv_heads * head_dim * tokens * bytes_per_elem * 2


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    description: str
    batch: int
    layers: int
    q_heads: int
    kv_heads: int
    head_dim: int
    max_seq_len: int
    top_k: int
    modes: tuple
    seed: int
    recipe: str                      # planting recipe, see _plant_*
    heavy: int                       # planted heavy positions (per head or per sequence)
    ragged: Optional[tuple] = None   # (lo, hi) inclusive per-sequence lengths
    heavy_keep: float = 1.0          # fraction of the heavy set kept layer to layer
    sinks: int = 0                   # attention-sink positions 0..sinks-1 (keys x3)

    @property
    def group(self) -> int:
        return self.q_heads // self.kv_heads

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny": Workload(
        name="tiny",
        description="batch 1, 4 attention-only layers (full, full+select, sparse, sparse), "
                    "8 query / 2 KV heads, d=128, N=4096, k=256, 64 heavy rows shared across layers",
        batch=1, layers=4, q_heads=8, kv_heads=2, head_dim=128, max_seq_len=4096, top_k=256,
        modes=(FULL, FULL_SELECT, SPARSE, SPARSE), seed=0, recipe="mean_of_heavy", heavy=64),
    "llama2-7b-10k": Workload(
        name="llama2-7b-10k",
        description="LLaMA-2-7B attention shape: batch 1, 32 layers, 32 heads MHA, d=128, "
                    "N=10240, k=512, selection at L2 and L7, 256 heavy positions per head",
        batch=1, layers=32, q_heads=32, kv_heads=32, head_dim=128, max_seq_len=10240, top_k=512,
        modes=figure2_schedule(32, 7), seed=1, recipe="direction", heavy=256),
    "llama3-8b-32k": Workload(
        name="llama3-8b-32k",
        description="LLaMA-3-8B attention shape: batch 4, 32 layers, 32 query / 8 KV heads, d=128, "
                    "N=32768, k=2048, selection at L2 and L14, 1024 heavy positions per sequence, "
                    "80% kept layer to layer",
        batch=4, layers=32, q_heads=32, kv_heads=8, head_dim=128, max_seq_len=32768, top_k=2048,
        modes=figure2_schedule(32, 14), seed=2, recipe="direction", heavy=1024, heavy_keep=0.8),
    "llama2-7b-100k": Workload(
        name="llama2-7b-100k",
        description="long-context LLaMA-2-7B shape: batch 1, 32 layers, 32 heads MHA, d=128, "
                    "N=102400, k=4096, selection at L2 and L7, 256 heavy per head, 4 sink tokens",
        batch=1, layers=32, q_heads=32, kv_heads=32, head_dim=128, max_seq_len=102400,
        top_k=4096, modes=figure2_schedule(32, 7), seed=3, recipe="direction", heavy=256, sinks=4),
    "serving-b32": Workload(
        name="serving-b32",
        description="batched serving: LLaMA-3-8B GQA shape, batch 32, N_max=16384, ragged lengths "
                    "uniform in [8192, 16384], selection at L2 and L14, 512 heavy per sequence",
        batch=32, layers=32, q_heads=32, kv_heads=8, head_dim=128, max_seq_len=16384, top_k=1024,
        modes=figure2_schedule(32, 14), seed=4, recipe="direction", heavy=512,
        ragged=(8192, 16384)),
}
SERVING_TOP_KS = (256, 1024, 4096)


def seq_lens(wl: Workload) -> np.ndarray:
    if wl.ragged is None:
        return np.full(wl.batch, wl.max_seq_len, dtype=np.int32)
    rs = np.random.RandomState(wl.seed + 1000)
    lo, hi = wl.ragged
    return rs.randint(lo, hi + 1, size=wl.batch).astype(np.int32)


def heavy_positions(wl: Workload) -> list:
    """Planted heavy positions: list over layers of int64 arrays [B, Hkv, heavy].

    "direction" recipes with MHA draw a set per head; GQA recipes draw one set
    per sequence and share it across the sequence's KV heads.  With
    heavy_keep < 1 each layer keeps that fraction of the previous layer's set
    and draws the rest afresh.  Sink positions are never heavy.
    """
    rs = np.random.RandomState(wl.seed + 2000)
    lens = seq_lens(wl)
    per_head = wl.q_heads == wl.kv_heads and wl.recipe == "direction"
    sets = []
    cur = None
    for layer in range(wl.layers):
        new = np.zeros((wl.batch, wl.kv_heads, wl.heavy), dtype=np.int64)
        for b in range(wl.batch):
            lo, hi = wl.sinks, int(lens[b])
            units = wl.kv_heads if per_head else 1
            for u in range(units):
                if cur is None:
                    chosen = rs.choice(np.arange(lo, hi), size=wl.heavy, replace=False)
                else:
                    prev = cur[b, u]
                    n_keep = int(round(wl.heavy * wl.heavy_keep))
                    if n_keep >= wl.heavy:
                        chosen = prev
                    else:
                        kept = rs.choice(prev, size=n_keep, replace=False)
                        pool = np.setdiff1d(np.arange(lo, hi), prev)
                        fresh = rs.choice(pool, size=wl.heavy - n_keep, replace=False)
                        chosen = np.concatenate([kept, fresh])
                if per_head:
                    new[b, u] = chosen
                else:
                    new[b, :] = chosen
        sets.append(new)
        cur = new
    return sets


def _layer_generator(wl: Workload, layer: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(wl.seed * 1_000_003 + layer * 7919 + 17)
    return g


def generate_layer(wl: Workload, layer: int, device="cpu", heavy=None):
    """(q [B,Hq,d], K [B,Hkv,Nmax,d], V [B,Hkv,Nmax,d]) in bf16 for one layer.

    Recipes:
      mean_of_heavy  K, V, z ~ N(0,1); q[h] = z + 0.5 * mean of the layer's K
                     rows at the heavy positions of KV head g(h).
      direction      K, V, z ~ N(0,1); a random unit vector u per (batch, KV
                     head) and layer; K[p] += 1.0 * u at heavy positions p;
                     q[h] = z + sqrt(d) * u_{g(h)}, so a heavy key's scaled
                     logit gains +1 on average.  Sink positions have K x 3.
    """
    if heavy is None:
        heavy = heavy_positions(wl)[layer]
    g = _layer_generator(wl, layer, device)
    B, Hq, Hkv, d, N = wl.batch, wl.q_heads, wl.kv_heads, wl.head_dim, wl.max_seq_len
    G = Hq // Hkv
    K = torch.randn((B, Hkv, N, d), generator=g, device=device, dtype=torch.float32)
    V = torch.randn((B, Hkv, N, d), generator=g, device=device, dtype=torch.float32)
    z = torch.randn((B, Hq, d), generator=g, device=device, dtype=torch.float32)
    hv = torch.as_tensor(heavy, device=device, dtype=torch.int64)           # [B,Hkv,h]
    rows = (torch.arange(B * Hkv, device=device).view(B, Hkv, 1) * N + hv).reshape(-1)
    if wl.recipe == "mean_of_heavy":
        Kb = K.to(torch.bfloat16).float()
        sel = Kb.view(B * Hkv * N, d).index_select(0, rows).view(B, Hkv, -1, d)
        mean = sel.mean(dim=2)                                              # [B,Hkv,d]
        q = z + 0.5 * mean.repeat_interleave(G, dim=1)
    elif wl.recipe == "direction":
        u = torch.randn((B, Hkv, d), generator=g, device=device, dtype=torch.float32)
        u = u / u.norm(dim=-1, keepdim=True)
        Kf = K.view(B * Hkv * N, d)
        bias = u.view(B * Hkv, 1, d).expand(B * Hkv, hv.shape[-1], d).reshape(-1, d)
        Kf.index_add_(0, rows, bias)
        if wl.sinks:
            K[:, :, : wl.sinks, :] *= 3.0
        q = z + math.sqrt(d) * u.repeat_interleave(G, dim=1)
    else:
        raise ValueError(wl.recipe)
    return q.to(torch.bfloat16), K.to(torch.bfloat16), V.to(torch.bfloat16)


def random_case(seed: int, batch: int, q_heads: int, kv_heads: int, max_seq_len: int,
                lens: Sequence[int], head_dim: int = 128, device="cpu", dist="normal"):
    """Plain random q/K/V for shape sweeps (no planting).  dist: 'normal' or
    'uniform_small' (integers in [-2, 2], exact in bf16)."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    shapes = [(batch, q_heads, head_dim), (batch, kv_heads, max_seq_len, head_dim),
              (batch, kv_heads, max_seq_len, head_dim)]
    if dist == "normal":
        out = [torch.randn(s, generator=g, device=device) for s in shapes]
    elif dist == "uniform_small":
        out = [torch.randint(-2, 3, s, generator=g, device=device).float() for s in shapes]
    else:
        raise ValueError(dist)
    q, K, V = (t.to(torch.bfloat16) for t in out)
    return q, K, V, torch.as_tensor(np.asarray(lens, dtype=np.int32))


def random_index_sets(seed: int, batch: int, kv_heads: int, k: int, lens: Sequence[int],
                      pad_fraction: float = 0.0) -> np.ndarray:
    """Distinct ascending positions per (b, kv head), -1 padded at the end.

    pad_fraction of the k slots (at least where len < k) are padding."""
    rs = np.random.RandomState(seed)
    idx = np.full((batch, kv_heads, k), -1, dtype=np.int32)
    for b in range(batch):
        n = int(lens[b])
        for g in range(kv_heads):
            live = min(k, n)
            live = max(0, min(live, int(round(k * (1.0 - pad_fraction)))) if pad_fraction else live)
            if live:
                sel = np.sort(rs.choice(n, size=live, replace=False))
                idx[b, g, :live] = sel
    return idx


def u16(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
