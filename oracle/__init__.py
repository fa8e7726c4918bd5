"""CPU oracle for the TidalDecode decode step -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference arm of ``bench.py`` may import this package.  The product path
(``sparse_attention_td_gb300``) never imports it, and it imports nothing from
the product: the two share only the seeded input generators in ``workloads``.

The arithmetic lives in ``td_oracle.c`` (plain loops, fp64); this module
compiles it with gcc and wraps it with ctypes for numpy arrays.  Inputs are
bf16 bit patterns held in ``numpy.uint16`` arrays.

What it computes (TidalDecode paper review page):
  * ``attend``       -- A = q K^T / sqrt(d), H = softmax(A) V (§三, PPSA formula)
  * ``group_scores`` -- the selection score of a KV head: sum of its query
                        heads' scaled logits (reading for grouped-query heads)
  * ``topk``         -- top-k positions, ties to the lower position (§二 core
                        insight; §三 Figure 2 "token selection -> top-k")
  * ``decode_group`` / ``decode_step`` -- the per-step schedule of Figure 2:
                        FULL, FULL_SELECT (full + selection), SPARSE (reuse
                        the persisted positions, §三 PPSA).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

MODE_FULL = 0
MODE_FULL_SELECT = 1
MODE_SPARSE = 2

OK = 0
ERR_ARG = 1
ERR_NO_SELECTION = 2
ERR_NOMEM = 3

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "td_oracle.c")
_lock = threading.Lock()
_cache: dict[int, "Oracle"] = {}


def lib_path(mutant: int = 0) -> str:
    name = "libtd_oracle.so" if mutant == 0 else f"libtd_oracle_mutant{mutant}.so"
    return os.path.join(_HERE, "_build", name)


def build(mutant: int = 0, force: bool = False) -> str:
    """Compile td_oracle.c (with OpenMP when gcc supports it) and return the .so path."""
    out = lib_path(mutant)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(_SRC)):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = f"{out}.{os.getpid()}.tmp"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", f"-DORACLE_MUTANT={mutant}", _SRC,
            "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:2] + ["-fopenmp"] + base[2:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, out)
    return out


def _u16(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("oracle inputs are bf16 bit patterns (numpy.uint16)")
    return a


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


class Oracle:
    """ctypes wrapper of one build of td_oracle.c."""

    def __init__(self, mutant: int = 0):
        self.mutant = mutant
        self._lib = ctypes.CDLL(build(mutant))
        L = self._lib
        u16p = ctypes.POINTER(ctypes.c_uint16)
        f64p = ctypes.POINTER(ctypes.c_double)
        i32p = ctypes.POINTER(ctypes.c_int32)
        L.oracle_bf16_to_double.restype = ctypes.c_double
        L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        L.oracle_logit.restype = ctypes.c_double
        L.oracle_logit.argtypes = [u16p, u16p, ctypes.c_int, ctypes.c_double]
        L.oracle_softmax.restype = None
        L.oracle_softmax.argtypes = [f64p, ctypes.c_int, f64p]
        L.oracle_attend.restype = ctypes.c_int
        L.oracle_attend.argtypes = [u16p, u16p, u16p, ctypes.c_int, i32p, ctypes.c_int,
                                    ctypes.c_double, f64p, f64p]
        L.oracle_group_scores.restype = None
        L.oracle_group_scores.argtypes = [u16p, ctypes.c_int, u16p, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_double, f64p]
        L.oracle_topk.restype = ctypes.c_int
        L.oracle_topk.argtypes = [f64p, ctypes.c_int, ctypes.c_int, i32p]
        vpp = ctypes.POINTER(ctypes.c_void_p)
        L.oracle_decode_group.restype = ctypes.c_int
        L.oracle_decode_group.argtypes = [ctypes.c_int, i32p, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                          vpp, vpp, vpp, i32p, ctypes.POINTER(ctypes.c_int),
                                          vpp, vpp]
        L.oracle_decode_step.restype = ctypes.c_int
        L.oracle_decode_step.argtypes = [ctypes.c_int] * 5 + [i32p, ctypes.c_int, i32p,
                                                              ctypes.c_int, ctypes.c_double,
                                                              vpp, vpp, vpp, vpp, i32p]
        L.oracle_index_overlap.restype = ctypes.c_int
        L.oracle_index_overlap.argtypes = [i32p, i32p, ctypes.c_int]
        L.oracle_coverage_count.restype = ctypes.c_int
        L.oracle_coverage_count.argtypes = [f64p, ctypes.c_int, ctypes.c_double, ctypes.c_int]
        L.oracle_mutant_id.restype = ctypes.c_int
        L.oracle_num_threads.restype = ctypes.c_int
        L.oracle_set_threads.restype = None
        L.oracle_set_threads.argtypes = [ctypes.c_int]

    # -- single pieces -------------------------------------------------------
    def bf16_to_double(self, bits: int) -> float:
        return self._lib.oracle_bf16_to_double(int(bits))

    def logit(self, q: np.ndarray, krow: np.ndarray, scale: float) -> float:
        q, krow = _u16(q), _u16(krow)
        return self._lib.oracle_logit(_ptr(q, ctypes.c_uint16), _ptr(krow, ctypes.c_uint16),
                                      q.shape[-1], scale)

    def softmax(self, a: np.ndarray) -> np.ndarray:
        a = np.ascontiguousarray(a, dtype=np.float64)
        p = np.zeros_like(a)
        self._lib.oracle_softmax(_ptr(a, ctypes.c_double), a.size, _ptr(p, ctypes.c_double))
        return p

    def attend(self, q, K, V, scale, rows=None, return_p=False):
        """out[d] (and optionally p) of one query head over K/V rows ([n][d])."""
        q, K, V = _u16(q), _u16(K), _u16(V)
        d = q.shape[-1]
        if rows is None:
            n = K.shape[0]
            rows_p = None
        else:
            rows = np.ascontiguousarray(rows, dtype=np.int32)
            n = rows.size
            rows_p = _ptr(rows, ctypes.c_int32)
        out = np.zeros(d, dtype=np.float64)
        p = np.zeros(max(n, 1), dtype=np.float64)
        rc = self._lib.oracle_attend(_ptr(q, ctypes.c_uint16), _ptr(K, ctypes.c_uint16),
                                     _ptr(V, ctypes.c_uint16), d, rows_p, n, scale,
                                     _ptr(out, ctypes.c_double), _ptr(p, ctypes.c_double))
        if rc:
            raise RuntimeError(f"oracle_attend failed: {rc}")
        return (out, p[:n]) if return_p else out

    def group_scores(self, q_group, K, n, scale) -> np.ndarray:
        q_group, K = _u16(q_group), _u16(K)
        G, d = q_group.shape
        s = np.zeros(max(n, 1), dtype=np.float64)
        self._lib.oracle_group_scores(_ptr(q_group, ctypes.c_uint16), G,
                                      _ptr(K, ctypes.c_uint16), d, n, scale,
                                      _ptr(s, ctypes.c_double))
        return s[:n]

    def topk(self, s: np.ndarray, k: int) -> np.ndarray:
        s = np.ascontiguousarray(s, dtype=np.float64)
        idx = np.full(max(k, 1), -7, dtype=np.int32)
        kept = self._lib.oracle_topk(_ptr(s, ctypes.c_double), s.size, k,
                                     _ptr(idx, ctypes.c_int32))
        if kept < 0:
            raise MemoryError("oracle_topk")
        return idx[:k]

    # -- schedules ------------------------------------------------------------
    def decode_group(self, modes, q_group, K, V, n_b, k, scale, idx_in=None):
        """One (batch row, KV head) through L layers.

        q_group: list of L arrays [G][d]; K, V: lists of L arrays [>=n_b][d].
        Returns (out [L][G][d] float64, idx_per_layer [L][k] int32 (rows of -2
        where a layer neither selected nor attended sparsely), final idx, rc).
        """
        L = len(modes)
        modes_a = np.ascontiguousarray(modes, dtype=np.int32)
        qs = [_u16(x) for x in q_group]
        Ks = [_u16(x) for x in K]
        Vs = [_u16(x) for x in V]
        G, d = qs[0].shape if L else (1, 128)
        outs = [np.zeros((G, d), dtype=np.float64) for _ in range(L)]
        per = [np.full(max(k, 1), -2, dtype=np.int32) for _ in range(L)]
        state = np.full(max(k, 1), -1, dtype=np.int32)
        valid = ctypes.c_int(0)
        if idx_in is not None:
            state[:k] = idx_in
            valid.value = 1

        def arr(lst):
            return (ctypes.c_void_p * max(L, 1))(*[x.ctypes.data for x in lst])

        rc = self._lib.oracle_decode_group(L, _ptr(modes_a, ctypes.c_int32), G, d, n_b, k, scale,
                                           arr(qs), arr(Ks), arr(Vs),
                                           _ptr(state, ctypes.c_int32), ctypes.byref(valid),
                                           arr(outs), arr(per))
        return (np.stack(outs) if L else np.zeros((0, G, d)),
                np.stack([p[:k] for p in per]) if L else np.zeros((0, k), np.int32),
                state[:k].copy(), rc)

    def decode_step(self, modes, q, K, V, seq_lens, k, scale):
        """Whole batched step.  q: list of L [B][Hq][d]; K, V: list of L
        [B][Hkv][Nmax][d] (uint16 bf16 bits).  Returns (out list of L
        [B][Hq][d] float64, idx_final [B][Hkv][k], rc)."""
        L = len(modes)
        qs = [_u16(x) for x in q]
        Ks = [_u16(x) for x in K]
        Vs = [_u16(x) for x in V]
        B, Hq, d = qs[0].shape
        Hkv, Nmax = Ks[0].shape[1], Ks[0].shape[2]
        outs = [np.zeros((B, Hq, d), dtype=np.float64) for _ in range(L)]
        idx = np.full((B, Hkv, max(k, 1)), -1, dtype=np.int32)
        sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
        modes_a = np.ascontiguousarray(modes, dtype=np.int32)

        def arr(lst):
            return (ctypes.c_void_p * max(L, 1))(*[x.ctypes.data for x in lst])

        rc = self._lib.oracle_decode_step(B, Hq, Hkv, d, Nmax, _ptr(sl, ctypes.c_int32), L,
                                          _ptr(modes_a, ctypes.c_int32), k, scale,
                                          arr(qs), arr(Ks), arr(Vs), arr(outs),
                                          _ptr(idx, ctypes.c_int32))
        return outs, idx[:, :, :k], rc

    def index_overlap(self, a, b) -> int:
        """Positions present in both sets (entries < 0 ignored)."""
        a = np.ascontiguousarray(a, dtype=np.int32)
        b = np.ascontiguousarray(b, dtype=np.int32)
        assert a.shape == b.shape and a.ndim == 1
        return int(self._lib.oracle_index_overlap(_ptr(a, ctypes.c_int32), _ptr(b, ctypes.c_int32),
                                               len(a)))

    def coverage_count(self, s, tau: float, k_max: int) -> int:
        """Smallest k whose top-k scores hold >= 1 - tau of softmax(s), <= k_max."""
        s = np.ascontiguousarray(s, dtype=np.float64)
        k = self._lib.oracle_coverage_count(_ptr(s, ctypes.c_double), s.size, float(tau),
                                            int(k_max))
        if k < 0:
            raise MemoryError("oracle_coverage_count")
        return int(k)

    def mutant_id(self) -> int:
        return self._lib.oracle_mutant_id()

    def set_threads(self, n: int) -> None:
        """Threads the OpenMP regions use from now on (1 = serial)."""
        self._lib.oracle_set_threads(int(n))

    def num_threads(self) -> int:
        return self._lib.oracle_num_threads()


def get(mutant: int = 0) -> Oracle:
    with _lock:
        if mutant not in _cache:
            _cache[mutant] = Oracle(mutant)
        return _cache[mutant]


def scale_for(d: int) -> float:
    """The softmax scale 1/sqrt(d) rounded to fp32, then widened (the kernel's constant)."""
    return float(np.float32(1.0) / np.sqrt(np.float32(d)))


def bf16_bits(x) -> np.ndarray:
    """Round a float array to bf16 (nearest-even) and return the bit patterns.

    Used by tests to build small exact inputs; values already representable in
    bf16 come back unchanged."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    rounding = ((u >> 16) & 1) + 0x7FFF
    return ((u + rounding) >> 16).astype(np.uint16)


def bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
