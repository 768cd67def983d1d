"""CPU oracle for paged decode / verify attention -- TEST INFRASTRUCTURE ONLY.

Only `tests/`, `__graft_entry__.smoke()` and the benchmark's CPU-baseline leg
may import this package.  The product path (the CUDA library and its Python
binding) never does, and this package shares no code with it: it decodes codes
with its own tables (in `pa_oracle.c`), plans work with its own rule
(`plan.py`) and merges split results with its own definition (`merge.py`).

Functions
---------
attention(w, rows=None, threads=None) -> (out[rows, Dv] float64, lse[rows])
    The exact definition, evaluated in double precision by `pa_oracle.c`.
row_ties(w, b, j, h, delta) -> (vmin, vmax, gap, count)
    Near-tie analysis of one row (INT8 / INT4 with large per-channel scales).
e4m3_table() -> float64[256]
max_abs_scale(k_scale) -> float
    max |k_scale| over (kv head, channel); 1.0 when that maximum is 0.
round_to(x, dtype) -> the same values rounded (RNE) to "f32" / "f16" / "bf16".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

from .merge import lse_merge  # noqa: F401
from .plan import plan  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")

_DT = {"f16": 0, "bf16": 1, "e4m3": 2, "int8": 3, "int4": 4}
_SM = {"none": 0, "tensor": 1, "channel": 2, "token": 3}
_ERR = {0: "ok", 1: "bad argument", 2: "block id out of range", 3: "out of memory"}


class _Problem(ctypes.Structure):
    _fields_ = [(k, ctypes.c_int32) for k in
                ("B", "n", "Hq", "Hkv", "Dk", "Dv", "bs", "num_blocks", "max_blocks_per_seq",
                 "q_dtype", "kv_dtype", "k_scale_mode", "v_scale_mode", "v_is_k_prefix", "causal")] + \
              [("softmax_scale", ctypes.c_double)]


_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile pa_oracle.c with the host C compiler (plain C11, -O2)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.POINTER
            lib.orc_attention.restype = ctypes.c_int
            lib.orc_attention.argtypes = [P(_Problem)] + [ctypes.c_void_p] * 3 + \
                [P(ctypes.c_int32), P(ctypes.c_int32), ctypes.c_void_p, ctypes.c_void_p,
                 P(ctypes.c_int32), ctypes.c_int64, P(ctypes.c_double), P(ctypes.c_double), ctypes.c_int]
            lib.orc_row_ties.restype = ctypes.c_int
            lib.orc_row_ties.argtypes = [P(_Problem)] + [ctypes.c_void_p] * 3 + \
                [P(ctypes.c_int32), P(ctypes.c_int32), ctypes.c_void_p, ctypes.c_void_p,
                 ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                 P(ctypes.c_double), P(ctypes.c_double), P(ctypes.c_double), P(ctypes.c_int32)]
            lib.orc_e4m3_table.restype = None
            lib.orc_e4m3_table.argtypes = [P(ctypes.c_double)]
            lib.orc_f16_value.restype = ctypes.c_double
            lib.orc_f16_value.argtypes = [ctypes.c_uint16]
            lib.orc_bf16_value.restype = ctypes.c_double
            lib.orc_bf16_value.argtypes = [ctypes.c_uint16]
            lib.orc_int4_value.restype = ctypes.c_double
            lib.orc_int4_value.argtypes = [ctypes.c_uint8, ctypes.c_int]
            _lib = lib
    return _lib


def _np(t, dtype=None):
    """CPU numpy view of a tensor / array (copies device tensors to host)."""
    if t is None:
        return None
    if hasattr(t, "detach"):
        t = t.detach()
        if t.device.type != "cpu":
            t = t.cpu()
        if dtype is None and str(t.dtype) in ("torch.float16", "torch.bfloat16"):
            import torch
            t = t.view(torch.int16)
        t = t.contiguous().numpy()
    a = np.ascontiguousarray(t)
    return a if dtype is None else np.ascontiguousarray(a, dtype=dtype)


def _problem(w) -> _Problem:
    return _Problem(B=w.B, n=w.n, Hq=w.Hq, Hkv=w.Hkv, Dk=w.Dk, Dv=w.Dv, bs=w.bs,
                    num_blocks=w.num_blocks, max_blocks_per_seq=w.max_blocks_per_seq,
                    q_dtype=_DT[w.q_dtype], kv_dtype=_DT[w.kv_dtype],
                    k_scale_mode=_SM[w.k_scale_mode], v_scale_mode=_SM[w.v_scale_mode],
                    v_is_k_prefix=int(bool(w.v_is_k_prefix)), causal=int(bool(w.causal)),
                    softmax_scale=float(w.softmax_scale))


class HostArrays:
    """Host copies of a workload's buffers, reusable across oracle calls."""

    def __init__(self, w):
        self.p = _problem(w)
        self.q = _np(w.q)
        self.k = _np(w.k_pool)
        self.v = _np(w.v_pool) if w.v_pool is not None else None
        self.table = _np(w.block_table, np.int32)
        self.lens = _np(w.context_lens, np.int32)
        self.ks = _np(w.k_scale, np.float32) if w.k_scale is not None else None
        self.vs = _np(w.v_scale, np.float32) if w.v_scale is not None else None
        self.B, self.n, self.Hq, self.Dv = w.B, w.n, w.Hq, w.Dv


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def attention(w, rows: Optional[Sequence[Sequence[int]]] = None, threads: Optional[int] = None,
              host: Optional[HostArrays] = None):
    """Exact paged attention for the given (b, j, h) rows (default: all rows,
    in (b, j, h) order).  Returns (out [num_rows, Dv] float64, lse [num_rows])."""
    lib = _load()
    H = host if host is not None else HostArrays(w)
    if rows is None:
        grid = np.stack(np.meshgrid(np.arange(H.B), np.arange(H.n), np.arange(H.Hq), indexing="ij"), -1)
        rows = grid.reshape(-1, 3)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 3))
    nr = rows.shape[0]
    out = np.zeros((nr, H.Dv), dtype=np.float64)
    lse = np.zeros((nr,), dtype=np.float64)
    if threads is None:
        threads = len(os.sched_getaffinity(0))
    P = ctypes.POINTER
    st = lib.orc_attention(ctypes.byref(H.p), _ptr(H.q), _ptr(H.k), _ptr(H.v),
                           H.table.ctypes.data_as(P(ctypes.c_int32)), H.lens.ctypes.data_as(P(ctypes.c_int32)),
                           _ptr(H.ks), _ptr(H.vs), rows.ctypes.data_as(P(ctypes.c_int32)), nr,
                           out.ctypes.data_as(P(ctypes.c_double)), lse.ctypes.data_as(P(ctypes.c_double)),
                           int(threads))
    if st != 0:
        raise ValueError(f"oracle: {_ERR.get(st, st)}")
    return out, lse


def row_ties(w, b: int, j: int, h: int, delta: float, host: Optional[HostArrays] = None):
    lib = _load()
    H = host if host is not None else HostArrays(w)
    vmin = np.zeros(H.Dv, dtype=np.float64)
    vmax = np.zeros(H.Dv, dtype=np.float64)
    gap = ctypes.c_double()
    cnt = ctypes.c_int32()
    P = ctypes.POINTER
    st = lib.orc_row_ties(ctypes.byref(H.p), _ptr(H.q), _ptr(H.k), _ptr(H.v),
                          H.table.ctypes.data_as(P(ctypes.c_int32)), H.lens.ctypes.data_as(P(ctypes.c_int32)),
                          _ptr(H.ks), _ptr(H.vs), b, j, h, float(delta),
                          vmin.ctypes.data_as(P(ctypes.c_double)), vmax.ctypes.data_as(P(ctypes.c_double)),
                          ctypes.byref(gap), ctypes.byref(cnt))
    if st != 0:
        raise ValueError(f"oracle: {_ERR.get(st, st)}")
    return vmin, vmax, gap.value, cnt.value


def e4m3_table() -> np.ndarray:
    lib = _load()
    t = np.zeros(256, dtype=np.float64)
    lib.orc_e4m3_table(t.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    return t


def f16_value(bits: int) -> float:
    return _load().orc_f16_value(bits)


def bf16_value(bits: int) -> float:
    return _load().orc_bf16_value(bits)


def int4_value(byte: int, high: int) -> float:
    return _load().orc_int4_value(byte, high)


def max_abs_scale(k_scale) -> float:
    """The fold normaliser of the onnxruntime PR #32520 page ("[CUDA] Normalize
    the PER_CHANNEL K scale folded into Q for paged XQA", Approach): the largest
    |k_scale| over every (kv head, channel) entry, taken as 1 when it is 0."""
    a = np.abs(_np(k_scale, np.float64))
    m = float(a.max()) if a.size else 0.0
    return 1.0 if m == 0.0 else m


def round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 values to f32 / f16 / bf16 (round to nearest even) and
    return them as float64."""
    import torch
    t = torch.from_numpy(np.asarray(x, dtype=np.float64))
    tgt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dtype]
    return t.to(tgt).to(torch.float64).numpy()
