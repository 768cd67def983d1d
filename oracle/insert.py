"""CPU oracle for the quantized paged KV insert -- TEST INFRASTRUCTURE ONLY.

Only `tests/`, `__graft_entry__.smoke()` and the benchmark's CPU-baseline leg
may use this module; the product path never does, and nothing here is shared
with it.

What it computes (the write that precedes paged attention): the next_n new
tokens of request b sit at logical positions L_b - next_n + j (j < next_n;
context_lens already count them, as for the attention).  Each new K / V row
of kv head g is quantized and stored at block block_table[b][pos / bs],
slot pos % bs, head-major inside the block; nothing else in the pool
changes.

Sources (page title, section):
  * onnxruntime PR #32520, "[CUDA] Normalize the PER_CHANNEL K scale folded
    into Q for paged XQA", Description: symmetric integer caches whose scale
    spans max|K| / 127 (INT8) or max|K| / 7 (INT4) -- codes are x / scale
    rounded, in [-127, 127] and [-7, 7].
  * CentML/vllm PR #167, "Q pad + KV insert", Design: the per-token
    quantization and paged insert of the new K/V rows, the only part of that
    op this library takes over (no RoPE, no Q padding).
  * 1Cat-vLLM PR #647, "Stop grouped-page4 null-block padding from leaking
    E4M3 NaN", Root cause: E4M3 (the "fn" format) has NaN at 0x7F / 0xFF and
    no infinity, so a finite value past 448 must saturate to 448.

Readings where the pages are silent: the quotient x / scale and the per-token scale max|x| / 448 are
formed in fp32 (the precision of the kernel; the pages fix none), then
rounded to nearest, ties to even: to the E4M3 grid saturating at +-448 (NaN
stays NaN), to an integer clamped to [-lim, lim] (NaN gives 0), or to
f16 / bf16 (IEEE: overflow gives inf).  A per-token scale that comes out 0
is replaced by 1.  A request whose length breaks the contract
(L_b < next_n, L_b > max_context_len, or more pages than table columns) is
flagged and left unwritten; a new token whose block id is outside
[1, num_blocks) is flagged and left unwritten.

Functions
---------
to_f32(x) -> float32 ndarray       exact value of f32 / f16 / bf16 inputs
e4m3_encode(y) -> uint8 codes       nearest E4M3 value, ties to the even code
int_encode(y, lim) -> int8 codes
f16_encode(y) / bf16_encode(y) -> uint16 bits
quantize_rows(x, kv_dtype, mode, scale) -> (row bytes uint8 [..., row_bytes],
                                            per-token scales or None)
insert(w, k_new, v_new) -> (k_pool, v_pool, flags)   new pools as uint8 arrays
"""
from __future__ import annotations

import numpy as np
import torch

from . import e4m3_table

ERR_BLOCK_ID = 0x1
ERR_CONTEXT_LEN = 0x2

_BITS = {"f16": 16, "bf16": 16, "e4m3": 8, "int8": 8, "int4": 4}
E4M3_MAX = 448.0


def _host(t):
    if t is None:
        return None
    if hasattr(t, "detach"):
        t = t.detach().cpu().contiguous()
        name = str(t.dtype)
        if name == "torch.bfloat16":
            return ("bf16", t.view(torch.int16).numpy().view(np.uint16))
        if name == "torch.float16":
            return ("f16", t.numpy())
        if name == "torch.float32":
            return ("f32", t.numpy())
        return ("raw", t.numpy())
    a = np.asarray(t)
    return ({np.dtype(np.float16): "f16", np.dtype(np.float32): "f32"}.get(a.dtype, "raw"), a)


def to_f32(x) -> np.ndarray:
    """Exact float32 values of an f32 / f16 / bf16 tensor or array (bf16 as
    its bits: the upper half of a float32)."""
    kind, a = _host(x)
    if kind == "f32":
        return a.astype(np.float32)
    if kind == "f16":
        return a.astype(np.float32)
    if kind == "bf16":
        return (a.astype(np.uint32) << 16).view(np.float32)
    raise TypeError("new K/V rows must be f32, f16 or bf16")


def e4m3_encode(y) -> np.ndarray:
    """Nearest E4M3 code of each fp32 value, ties to the even code (the code's
    last bit is the mantissa's), saturating to +-448; NaN gives 0x7F; the sign
    is kept, so negative values that round to zero give 0x80."""
    y = np.asarray(y, dtype=np.float32)
    a = np.abs(y.astype(np.float64))
    table = e4m3_table()
    pos = table[: 0x7F]                     # codes 0x00..0x7E: 0 .. 448, increasing
    lo = np.clip(np.searchsorted(pos, a, side="right") - 1, 0, 0x7E)
    hi = np.minimum(lo + 1, 0x7E)
    with np.errstate(invalid="ignore"):
        d_lo = a - pos[lo]
        d_hi = pos[hi] - a
        up = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0) & (hi != lo))
    code = np.where(up, hi, lo)
    code = np.where(a >= E4M3_MAX, 0x7E, code)          # saturate (inf included)
    code = code | np.where(np.signbit(y), 0x80, 0)
    code = np.where(np.isnan(y), 0x7F, code)
    return code.astype(np.uint8)


def int_encode(y, lim: int) -> np.ndarray:
    """round(y) to nearest, ties to even, clamped to [-lim, lim]; NaN gives 0."""
    y = np.asarray(y, dtype=np.float32)
    r = np.clip(np.rint(y), -lim, lim)
    r = np.where(np.isnan(y), 0, r)
    return r.astype(np.int8)


def f16_encode(y) -> np.ndarray:
    """IEEE half bits of each fp32 value (round to nearest even)."""
    with np.errstate(over="ignore"):
        return np.asarray(y, dtype=np.float32).astype(np.float16).view(np.uint16)


def bf16_encode(y) -> np.ndarray:
    """bfloat16 bits of each fp32 value: the upper 16 bits after rounding the
    lower 16 to nearest, ties to even (overflow carries into inf); NaN keeps a
    quiet NaN."""
    y = np.asarray(y, dtype=np.float32)
    u = y.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    return np.where(np.isnan(y), ((u >> 16).astype(np.uint16) | 0x0040), r).astype(np.uint16)


def quantize_rows(x: np.ndarray, kv_dtype: str, mode: str, scale=None):
    """Quantize rows x[..., D] (fp32 values) to the bytes the pool stores.

    mode "none": codes of x itself; "tensor": of x / scale (one fp32);
    "channel": of x / scale[d] (scale [D] fp32, broadcast over the rows);
    "token" (E4M3 only): s = max_d |x| / 448 per row (1 when that is 0), codes
    of x / s, and s is returned as the row's scale.  Returns (row bytes
    [..., D * bits / 8] uint8, per-row scales float32 or None)."""
    x = np.asarray(x, dtype=np.float32)
    tok = None
    if mode == "none":
        y = x
    elif mode == "tensor":
        y = x / np.float32(np.asarray(scale, dtype=np.float32).reshape(-1)[0])
    elif mode == "channel":
        y = x / np.asarray(scale, dtype=np.float32)
    elif mode == "token":
        if kv_dtype != "e4m3":
            raise ValueError("per-token scales are computed for E4M3 codes only")
        m = np.max(np.abs(x), axis=-1) if x.shape[-1] else np.zeros(x.shape[:-1], np.float32)
        s = (m.astype(np.float32) / np.float32(E4M3_MAX)).astype(np.float32)
        s = np.where(s == 0, np.float32(1.0), s).astype(np.float32)
        tok = s
        y = x / s[..., None]
    else:
        raise ValueError(mode)
    y = np.asarray(y, dtype=np.float32)
    if kv_dtype == "f16":
        data = f16_encode(y).view(np.uint8)
    elif kv_dtype == "bf16":
        data = np.ascontiguousarray(bf16_encode(y)).view(np.uint8)
    elif kv_dtype == "e4m3":
        data = e4m3_encode(y)
    elif kv_dtype == "int8":
        data = int_encode(y, 127).view(np.uint8)
    elif kv_dtype == "int4":
        c = int_encode(y, 7).astype(np.int16) & 0xF
        data = (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)
    else:
        raise ValueError(kv_dtype)
    return np.ascontiguousarray(data), tok


def insert(w, k_new, v_new=None, in_place: bool = False):
    """The pools after writing the new rows of every request.

    w: a workload (its pools, table, lengths, scales, shapes).  k_new: new K
    rows [B, n, Hkv, Dk] (f32 / f16 / bf16); v_new likewise with Dv (None
    when V is the first Dv channels of the K plane).  Returns (k_pool,
    v_pool or None, flags): uint8 arrays [num_blocks, block bytes] and the
    error bits the contract checks raise.  With in_place, w's pools must be
    numpy uint8 arrays and are written and returned instead of copies."""
    B, n, Hkv, bs = w.B, w.n, w.Hkv, w.bs
    table = np.asarray(w.block_table.cpu().numpy() if hasattr(w.block_table, "cpu") else w.block_table)
    lens = np.asarray(w.context_lens.cpu().numpy() if hasattr(w.context_lens, "cpu") else w.context_lens)
    flags = 0

    def plane(pool, new, D, mode, scale):
        nonlocal flags
        if pool is None:
            return None
        if in_place:
            out = pool
        else:
            out = np.array(pool.cpu().numpy() if hasattr(pool, "cpu") else pool, dtype=np.uint8, copy=True)
        x = to_f32(new).reshape(B, n, Hkv, D)
        row = D * _BITS[w.kv_dtype] // 8
        codes_bytes = Hkv * bs * row
        sc = None if scale is None else to_f32(scale)
        for b in range(B):
            L = int(lens[b])
            if L < n or L > w.max_context_len or (L + bs - 1) // bs > w.max_blocks_per_seq:
                flags |= ERR_CONTEXT_LEN
                continue
            for j in range(n):
                pos = L - n + j
                blk = int(table[b, pos // bs])
                slot = pos % bs
                if blk < 1 or blk >= w.num_blocks:
                    flags |= ERR_BLOCK_ID
                    continue
                for g in range(Hkv):
                    s = None
                    if mode == "tensor":
                        s = sc.reshape(-1)[:1]
                    elif mode == "channel":
                        s = sc.reshape(Hkv, -1)[g, :D]
                    data, tok = quantize_rows(x[b, j, g], w.kv_dtype, mode, s)
                    o = (g * bs + slot) * row
                    out[blk, o: o + row] = data
                    if tok is not None:
                        t = codes_bytes + (g * bs + slot) * 4
                        out[blk, t: t + 4] = np.asarray(tok, dtype=np.float32).reshape(1).view(np.uint8)
        return out

    kp = plane(w.k_pool, k_new, w.Dk, w.k_scale_mode, w.k_scale)
    vp = None
    if not w.v_is_k_prefix:
        vp = plane(w.v_pool, v_new, w.Dv, w.v_scale_mode, w.v_scale)
    return kp, vp, flags
