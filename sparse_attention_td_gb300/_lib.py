"""ctypes binding of libtd.so: argument marshalling and buffer checks only."""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

MODE_FULL = 0
MODE_FULL_SELECT = 1
MODE_SPARSE = 2
FLAG_INDEX_OUT_OF_RANGE = 0x1
FLAG_SEQ_LEN_OUT_OF_RANGE = 0x2
FLAG_WAIT_TIMEOUT = 0x4
NOALLOC_SCRATCH_BYTES = 8 << 20  # TD_NOALLOC_SCRATCH_BYTES: td_sparse_attn_noalloc's fixed scratch

_HERE = os.path.dirname(os.path.abspath(__file__))


def lib_path() -> str:
    return os.path.join(_HERE, "libtd.so")


class TdError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {td_status_string(status)} ({status})")


class Shape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("max_seq_len", ctypes.c_int32), ("scale", ctypes.c_float)]

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads


def default_scale(head_dim: int) -> float:
    """The library's scale when Shape.scale == 0: 1/sqrtf(head_dim) in fp32."""
    import numpy as np
    return float(np.float32(1.0) / np.sqrt(np.float32(head_dim)))


def make_shape(batch, num_q_heads, num_kv_heads, max_seq_len, head_dim=128, scale=0.0) -> Shape:
    return Shape(batch, num_q_heads, num_kv_heads, head_dim, max_seq_len, scale)


_lib = None


def lib():
    """Load libtd.so; raise if it has not been built (no fallback exists)."""
    global _lib
    if _lib is not None:
        return _lib
    path = lib_path()
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with `python -c \"import __graft_entry__ "
                          f"as g; g.build()\"` (or sparse_attention_td_gb300/build.py)")
    L = ctypes.CDLL(path)
    vp, sz, i32, u32p = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.POINTER(ctypes.c_uint32)
    shp = ctypes.POINTER(Shape)
    vpp = ctypes.POINTER(ctypes.c_void_p)
    L.td_status_string.restype = ctypes.c_char_p
    L.td_status_string.argtypes = [ctypes.c_int]
    L.td_workspace_size.restype = sz
    L.td_workspace_size.argtypes = [shp, i32]
    L.td_workspace_init.restype = ctypes.c_int
    L.td_workspace_init.argtypes = [vp, sz, vp]
    L.td_workspace_status.restype = ctypes.c_int
    L.td_workspace_status.argtypes = [vp, sz, u32p, vp]
    L.td_full_attn_select.restype = ctypes.c_int
    L.td_full_attn_select.argtypes = [shp, vp, vp, vp, vp, i32, vp, vp, vp, vp, vp, sz, vp]
    L.td_topk_select.restype = ctypes.c_int
    L.td_topk_select.argtypes = [shp, vp, vp, i32, vp, vp, sz, vp]
    L.td_full_attn_select_coverage.restype = ctypes.c_int
    L.td_full_attn_select_coverage.argtypes = [shp, vp, vp, vp, vp, ctypes.c_float, i32, vp, vp,
                                               vp, vp, vp, vp, sz, vp]
    L.td_probe_layer_reads.restype = ctypes.c_int
    L.td_probe_layer_reads.argtypes = [shp, vp, vp, vp, vp, i32, vp, i32, vp]
    L.td_kv_append.restype = ctypes.c_int
    L.td_kv_append.argtypes = [shp, vp, vp, vp, vp, vp, vp]
    L.td_decode_step_append.restype = ctypes.c_int
    L.td_decode_step_append.argtypes = [shp, i32, vp, vpp, vpp, vpp, vpp, vpp, vp, i32, vp, i32,
                                        vpp, vpp, vp, sz, vp, vpp]
    L.td_plan_create_append.restype = ctypes.c_int
    L.td_plan_create_append.argtypes = [ctypes.POINTER(vp), shp, i32, vp, vpp, vpp, vpp, vpp, vpp,
                                        vp, i32, vp, i32, vpp, vpp, vp, sz]
    L.td_plan_create_host.restype = ctypes.c_int
    L.td_plan_create_host.argtypes = [ctypes.POINTER(vp), shp, i32, vp, vp, vp, vpp, vpp, vp,
                                      i32, vp, i32, vp, vpp, vp, vp, sz]
    L.td_index_overlap.restype = ctypes.c_int
    L.td_index_overlap.argtypes = [shp, vp, vp, i32, vp, vp]
    L.td_sparse_attn.restype = ctypes.c_int
    L.td_sparse_attn.argtypes = [shp, vp, vp, vp, vp, vp, i32, vp, vp, vp, sz, vp]
    L.td_sparse_attn_noalloc.restype = ctypes.c_int
    L.td_sparse_attn_noalloc.argtypes = [shp, vp, vp, vp, vp, vp, i32, vp, vp, vp]
    L.td_decode_step.restype = ctypes.c_int
    L.td_decode_step.argtypes = [shp, i32, vp, vpp, vpp, vpp, vp, i32, vp, i32, vpp, vpp, vp, sz,
                                 vp, vpp]
    L.td_plan_create.restype = ctypes.c_int
    L.td_plan_create.argtypes = [ctypes.POINTER(vp), shp, i32, vp, vpp, vpp, vpp, vp, i32, vp, i32,
                                 vpp, vpp, vp, sz]
    L.td_plan_launch.restype = ctypes.c_int
    L.td_plan_launch.argtypes = [vp, vp]
    L.td_plan_destroy.restype = None
    L.td_plan_destroy.argtypes = [vp]
    L.td_set_tuning.restype = ctypes.c_int
    L.td_set_tuning.argtypes = [ctypes.c_char_p, i32]
    L.td_query_splits.restype = i32
    L.td_query_splits.argtypes = [shp, i32, i32]
    L.td_kernel_name.restype = ctypes.c_char_p
    L.td_kernel_name.argtypes = [shp, i32, i32]
    _lib = L
    return L


def td_status_string(status: int) -> str:
    return lib().td_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != 0:
        raise TdError(status, where)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _torch_stream(stream):
    if stream is None:
        return torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return stream
    return torch.cuda.ExternalStream(int(stream))


def _dev(t: Optional[torch.Tensor], name: str, dtype, numel: Optional[int] = None,
         optional=False) -> Optional[int]:
    if t is None:
        if optional:
            return None
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name} holds {t.numel()} elements, needs {numel}")
    return t.data_ptr()


def td_workspace_size(shape: Shape, top_k: int) -> int:
    return int(lib().td_workspace_size(ctypes.byref(shape), int(top_k)))


def td_workspace_init(ws: torch.Tensor, stream=None):
    _check(lib().td_workspace_init(_dev(ws, "ws", torch.uint8), ws.numel(), _stream(stream)),
           "td_workspace_init")


def td_workspace_status(ws: torch.Tensor, stream=None) -> int:
    flags = ctypes.c_uint32(0)
    _check(lib().td_workspace_status(_dev(ws, "ws", torch.uint8), ws.numel(),
                                     ctypes.byref(flags), _stream(stream)),
           "td_workspace_status")
    return flags.value


class Workspace:
    """A zero-initialised device workspace of td_workspace_size bytes."""

    def __init__(self, shape: Shape, top_k: int, device=None, stream=None):
        n = td_workspace_size(shape, top_k)
        if n == 0:
            raise TdError(1, "td_workspace_size")
        self.tensor = torch.empty(n, dtype=torch.uint8, device=device or "cuda")
        td_workspace_init(self.tensor, stream)

    @property
    def ptr(self) -> int:
        return self.tensor.data_ptr()

    @property
    def nbytes(self) -> int:
        return self.tensor.numel()

    def status(self, stream=None) -> int:
        return td_workspace_status(self.tensor, stream)


def _sizes(shape: Shape):
    B, Hq, Hkv, d, N = (shape.batch, shape.num_q_heads, shape.num_kv_heads, shape.head_dim,
                        shape.max_seq_len)
    return B * Hq * d, B * Hkv * N * d, B


def td_full_attn_select(shape: Shape, q, k_cache, v_cache, seq_lens, top_k, idx_out, out,
                        out_f32=None, scores_out=None, ws: Workspace = None, stream=None):
    nq, nkv, nb = _sizes(shape)
    st = lib().td_full_attn_select(
        ctypes.byref(shape), _dev(q, "q", torch.bfloat16, nq),
        _dev(k_cache, "k_cache", torch.bfloat16, nkv), _dev(v_cache, "v_cache", torch.bfloat16, nkv),
        _dev(seq_lens, "seq_lens", torch.int32, nb), int(top_k),
        _dev(idx_out, "idx_out", torch.int32, nb * shape.num_kv_heads * top_k, optional=top_k == 0),
        _dev(out, "out", torch.bfloat16, nq), _dev(out_f32, "out_f32", torch.float32, nq, True),
        _dev(scores_out, "scores_out", torch.float32, nkv // shape.head_dim, True),
        ws.ptr, ws.nbytes, _stream(stream))
    _check(st, "td_full_attn_select")


def td_full_attn_select_coverage(shape: Shape, q, k_cache, v_cache, seq_lens, tau, k_max, idx_out,
                                 counts_out, out, out_f32=None, scores_out=None,
                                 ws: Workspace = None, stream=None):
    nq, nkv, nb = _sizes(shape)
    st = lib().td_full_attn_select_coverage(
        ctypes.byref(shape), _dev(q, "q", torch.bfloat16, nq),
        _dev(k_cache, "k_cache", torch.bfloat16, nkv), _dev(v_cache, "v_cache", torch.bfloat16, nkv),
        _dev(seq_lens, "seq_lens", torch.int32, nb), float(tau), int(k_max),
        _dev(idx_out, "idx_out", torch.int32, nb * shape.num_kv_heads * k_max),
        _dev(counts_out, "counts_out", torch.int32, nb * shape.num_kv_heads, True),
        _dev(out, "out", torch.bfloat16, nq), _dev(out_f32, "out_f32", torch.float32, nq, True),
        _dev(scores_out, "scores_out", torch.float32, nkv // shape.head_dim, True),
        ws.ptr, ws.nbytes, _stream(stream))
    _check(st, "td_full_attn_select_coverage")


def td_topk_select(shape: Shape, scores, seq_lens, top_k, idx_out, ws: Workspace = None,
                   stream=None):
    nq, nkv, nb = _sizes(shape)
    st = lib().td_topk_select(
        ctypes.byref(shape), _dev(scores, "scores", torch.float32, nkv // shape.head_dim),
        _dev(seq_lens, "seq_lens", torch.int32, nb), int(top_k),
        _dev(idx_out, "idx_out", torch.int32, nb * shape.num_kv_heads * top_k),
        ws.ptr, ws.nbytes, _stream(stream))
    _check(st, "td_topk_select")


def td_index_overlap(shape: Shape, idx_a, idx_b, top_k, counts, stream=None):
    n = shape.batch * shape.num_kv_heads
    st = lib().td_index_overlap(
        ctypes.byref(shape), _dev(idx_a, "idx_a", torch.int32, n * top_k),
        _dev(idx_b, "idx_b", torch.int32, n * top_k), int(top_k),
        _dev(counts, "counts", torch.int32, n), _stream(stream))
    _check(st, "td_index_overlap")


def td_sparse_attn(shape: Shape, q, k_cache, v_cache, seq_lens, idx, top_k, out, out_f32=None,
                   ws: Workspace = None, stream=None):
    nq, nkv, nb = _sizes(shape)
    st = lib().td_sparse_attn(
        ctypes.byref(shape), _dev(q, "q", torch.bfloat16, nq),
        _dev(k_cache, "k_cache", torch.bfloat16, nkv), _dev(v_cache, "v_cache", torch.bfloat16, nkv),
        _dev(seq_lens, "seq_lens", torch.int32, nb),
        _dev(idx, "idx", torch.int32, nb * shape.num_kv_heads * top_k), int(top_k),
        _dev(out, "out", torch.bfloat16, nq), _dev(out_f32, "out_f32", torch.float32, nq, True),
        ws.ptr, ws.nbytes, _stream(stream))
    _check(st, "td_sparse_attn")


def td_sparse_attn_noalloc(shape: Shape, q, k_cache, v_cache, seq_lens, idx, top_k, out,
                           out_f32=None, stream=None):
    """td_sparse_attn without a workspace, for callers that cannot allocate
    device memory (scratch lives in a fixed array in the library)."""
    nq, nkv, nb = _sizes(shape)
    st = lib().td_sparse_attn_noalloc(
        ctypes.byref(shape), _dev(q, "q", torch.bfloat16, nq),
        _dev(k_cache, "k_cache", torch.bfloat16, nkv), _dev(v_cache, "v_cache", torch.bfloat16, nkv),
        _dev(seq_lens, "seq_lens", torch.int32, nb),
        _dev(idx, "idx", torch.int32, nb * shape.num_kv_heads * top_k), int(top_k),
        _dev(out, "out", torch.bfloat16, nq), _dev(out_f32, "out_f32", torch.float32, nq, True),
        _stream(stream))
    _check(st, "td_sparse_attn_noalloc")


def _ptr_array(tensors, name, dtype, numel, optional=False):
    ptrs = [_dev(t, f"{name}[{i}]", dtype, numel, optional) or 0 for i, t in enumerate(tensors)]
    return (ctypes.c_void_p * max(len(ptrs), 1))(*ptrs)


class _StepArgs:
    """Marshalled arguments of one decode step (kept alive while in use)."""

    def __init__(self, shape, modes, q, k_caches, v_caches, seq_lens, top_k, idx_buf, outs,
                 outs_f32, k_new=None, v_new=None):
        nq, nkv, nb = _sizes(shape)
        L = len(modes)
        if not (len(q) == len(k_caches) == len(v_caches) == len(outs) == L):
            raise ValueError("per-layer lists must have one entry per mode")
        if outs_f32 is not None and len(outs_f32) != L:
            raise ValueError("outs_f32 must have one entry per mode")
        self.L = L
        self.modes = (ctypes.c_int32 * max(L, 1))(*[int(m) for m in modes])
        self.q = _ptr_array(q, "q", torch.bfloat16, nq)
        self.k = _ptr_array(k_caches, "k_caches", torch.bfloat16, nkv)
        self.v = _ptr_array(v_caches, "v_caches", torch.bfloat16, nkv)
        self.outs = _ptr_array(outs, "outs", torch.bfloat16, nq)
        self.outs_f32 = (_ptr_array(outs_f32, "outs_f32", torch.float32, nq, optional=True)
                         if outs_f32 is not None else None)
        self.seq = _dev(seq_lens, "seq_lens", torch.int32, nb)
        needs_idx = any(int(m) != MODE_FULL for m in modes)
        self.idx = _dev(idx_buf, "idx_buf", torch.int32, nb * shape.num_kv_heads * top_k,
                        optional=not needs_idx)
        self.top_k = int(top_k)
        if (k_new is None) != (v_new is None):
            raise ValueError("k_new and v_new go together")
        self.append = k_new is not None
        if self.append:
            if not (len(k_new) == len(v_new) == L):
                raise ValueError("k_new / v_new need one entry per mode")
            n_new = nb * shape.num_kv_heads * shape.head_dim
            self.k_new = _ptr_array(k_new, "k_new", torch.bfloat16, n_new)
            self.v_new = _ptr_array(v_new, "v_new", torch.bfloat16, n_new)


def td_probe_layer_reads(shape: Shape, k_cache, v_cache, seq_lens, idx, top_k, sink,
                         stream=None):
    """Measurement aid: the K/V reads of one full (idx None) or sparse layer only."""
    nq, nkv, nb = _sizes(shape)
    st = lib().td_probe_layer_reads(
        ctypes.byref(shape), _dev(k_cache, "k_cache", torch.bfloat16, nkv),
        _dev(v_cache, "v_cache", torch.bfloat16, nkv), _dev(seq_lens, "seq_lens", torch.int32, nb),
        _dev(idx, "idx", torch.int32, nb * shape.num_kv_heads * max(int(top_k), 1), True),
        int(top_k), _dev(sink, "sink", torch.int32, 1), int(sink.numel()), _stream(stream))
    _check(st, "td_probe_layer_reads")


def td_kv_append(shape: Shape, k_cache, v_cache, k_new, v_new, seq_lens, stream=None):
    nq, nkv, nb = _sizes(shape)
    n_new = nb * shape.num_kv_heads * shape.head_dim
    st = lib().td_kv_append(
        ctypes.byref(shape), _dev(k_cache, "k_cache", torch.bfloat16, nkv),
        _dev(v_cache, "v_cache", torch.bfloat16, nkv), _dev(k_new, "k_new", torch.bfloat16, n_new),
        _dev(v_new, "v_new", torch.bfloat16, n_new), _dev(seq_lens, "seq_lens", torch.int32, nb),
        _stream(stream))
    _check(st, "td_kv_append")


def td_decode_step(shape: Shape, modes: Sequence[int], q, k_caches, v_caches, seq_lens, top_k,
                   idx_buf, outs, outs_f32=None, ws: Workspace = None, idx_valid=False,
                   stream=None, layer_events: Optional[Sequence] = None, k_new=None, v_new=None):
    """One decode step; with k_new / v_new (per-layer [B][Hkv][128] rows) the
    step also appends the new token to each layer's cache (td_decode_step_append)."""
    a = _StepArgs(shape, modes, q, k_caches, v_caches, seq_lens, top_k, idx_buf, outs, outs_f32,
                  k_new, v_new)
    ev = None
    if layer_events is not None:
        if len(layer_events) != a.L + 1:
            raise ValueError("layer_events needs num_layers + 1 events")
        for e in layer_events:
            if int(e.cuda_event) == 0:   # torch creates the CUDA event on first record
                e.record(_torch_stream(stream))
        ev =(ctypes.c_void_p * (a.L + 1))(*[int(e.cuda_event) for e in layer_events])
    if a.append:
        st = lib().td_decode_step_append(ctypes.byref(shape), a.L, a.modes, a.q, a.k, a.v, a.k_new,
                                         a.v_new, a.seq, a.top_k, a.idx, int(bool(idx_valid)),
                                         a.outs, a.outs_f32, ws.ptr, ws.nbytes, _stream(stream), ev)
        _check(st, "td_decode_step_append")
        return
    st = lib().td_decode_step(ctypes.byref(shape), a.L, a.modes, a.q, a.k, a.v, a.seq, a.top_k,
                              a.idx, int(bool(idx_valid)), a.outs, a.outs_f32, ws.ptr, ws.nbytes,
                              _stream(stream), ev)
    _check(st, "td_decode_step")


def _one_buffer(ts, name, n):
    """Device pointer of per-layer tensors that are consecutive slices of one
    buffer (layer l at the start + l * n values)."""
    base = ts[0].data_ptr()
    for l, t in enumerate(ts):
        if not t.is_cuda or t.dtype != torch.bfloat16 or t.numel() != n or \
                t.data_ptr() != base + 2 * n * l:
            raise ValueError(f"{name}: the layers must be consecutive slices of one bf16 buffer")
    return base


def _host_buffer(t, name, n):
    if t is None or t.is_cuda or t.dtype != torch.bfloat16 or t.numel() != n or \
            not t.is_contiguous():
        raise ValueError(f"{name}: one contiguous bf16 host tensor of {n} values expected")
    if not t.is_pinned():
        raise ValueError(f"{name}: the host tensor must be page-locked (pin_memory())")
    return t.data_ptr()


class Plan:
    """A decode step captured once into a CUDA graph (td_plan_create).  With
    q_host / out_host (page-locked host tensors of all layers' rows, [L][B][Hq][128])
    the step also copies the q rows in and the outputs back
    (td_plan_create_host); q and outs must then be slices of one device
    buffer each."""

    def __init__(self, shape: Shape, modes, q, k_caches, v_caches, seq_lens, top_k, idx_buf, outs,
                 outs_f32=None, ws: Workspace = None, idx_valid=False, k_new=None, v_new=None,
                 q_host=None, out_host=None):
        self._args = _StepArgs(shape, modes, q, k_caches, v_caches, seq_lens, top_k, idx_buf,
                               outs, outs_f32, k_new, v_new)
        self._keep = (q, k_caches, v_caches, seq_lens, idx_buf, outs, outs_f32, ws, k_new, v_new,
                      q_host, out_host)
        self._plan = ctypes.c_void_p(0)
        a = self._args
        if q_host is not None or out_host is not None:
            if a.append:
                raise ValueError("host q/out and KV append are separate plans")
            n = shape.batch * shape.num_q_heads * shape.head_dim
            qh = _host_buffer(q_host, "q_host", a.L * n)
            oh = _host_buffer(out_host, "out_host", a.L * n)
            st = lib().td_plan_create_host(
                ctypes.byref(self._plan), ctypes.byref(shape), a.L, a.modes, qh,
                _one_buffer(q, "q", n), a.k, a.v, a.seq, a.top_k, a.idx, int(bool(idx_valid)),
                _one_buffer(outs, "outs", n), a.outs_f32, oh, ws.ptr, ws.nbytes)
            _check(st, "td_plan_create_host")
            return
        if a.append:
            st = lib().td_plan_create_append(
                ctypes.byref(self._plan), ctypes.byref(shape), a.L, a.modes, a.q, a.k, a.v,
                a.k_new, a.v_new, a.seq, a.top_k, a.idx, int(bool(idx_valid)), a.outs, a.outs_f32,
                ws.ptr, ws.nbytes)
            _check(st, "td_plan_create_append")
            return
        st = lib().td_plan_create(ctypes.byref(self._plan), ctypes.byref(shape), a.L, a.modes,
                                  a.q, a.k, a.v, a.seq, a.top_k, a.idx, int(bool(idx_valid)),
                                  a.outs, a.outs_f32, ws.ptr, ws.nbytes)
        _check(st, "td_plan_create")

    def launch(self, stream=None):
        _check(lib().td_plan_launch(self._plan, _stream(stream)), "td_plan_launch")

    def close(self):
        if self._plan:
            lib().td_plan_destroy(self._plan)
            self._plan = ctypes.c_void_p(0)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def td_set_tuning(key: str, value: int):
    _check(lib().td_set_tuning(key.encode(), int(value)), f"td_set_tuning({key})")


def td_query_splits(shape: Shape, top_k: int, sparse: bool) -> int:
    return int(lib().td_query_splits(ctypes.byref(shape), int(top_k), int(bool(sparse))))


def td_kernel_name(shape: Shape, top_k: int, sparse: bool) -> str:
    return lib().td_kernel_name(ctypes.byref(shape), int(top_k), int(bool(sparse))).decode()
