"""CPU oracle for FP4 (MXFP4) paged MQA logits -- TEST INFRASTRUCTURE ONLY.

Only `tests/`, `__graft_entry__.smoke()` and the benchmark's CPU-baseline leg
may import this module; the product path never does.  It shares no code with
the CUDA library: the E2M1 and UE8M0 decoders below are written from the
formats' definitions, and every step is evaluated in float64.

Source: FlashInfer docs, "flashinfer.fp4_paged_mqa_logits", Parameters:
  q         [B, next_n, H, D/2] uint8, two E2M1 values per byte;
  sf_q      [B, next_n, H] int32, D/sf_vec_size UE8M0 scale bytes per
            (token, head), one per sf_vec_size consecutive values;
  kv_fused  [num_blocks, block_size, 1, D/2 + D/sf_vec_size] uint8: within a
            block, all tokens' packed values first, then all tokens' scale
            bytes (token order, or the page's interleaved order);
  weights   [B * next_n, H] float32 per-head weights;
  context_lens, block_table, max_context_len as for paged attention;
  output    [B * next_n, max_context_len] logits.

What it computes, per query row r = b * next_n + j and token t < vis:
    q^[h, d] = e2m1(q[b, j, h, d]) * 2^(sf_q byte of d's group - 127)
    k^[t, d] = e2m1(K[block_table[b][t / bs], t % bs, d]) * 2^(scale byte - 127)
    logit[r, t] = sum_h weights[r, h] * f(q^[h, :] . k^[t, :])
with f the identity (the page prints no formula: a plain weighted sum over
heads of the per-head dot products is the reading taken) or, with
rectify=True, max(0, .) per head.  vis = L_b for every row, or
L_b - (next_n - 1 - j) with causal=True.  Columns vis .. max_context_len - 1
are -inf.  Parity unpinned against the page for how heads combine (the page
does not print it); everything else is pinned by the tests.

Readings where the page is silent:
  - E2M1 packing: value 2i in the low nibble of byte i (as for INT4 KV);
  - UE8M0: 2^(e - 127), the byte 0xFF is NaN (no zero, no sign);
  - sf_q packing: byte i of the little-endian int32 scales values
    [i * sf_vec_size, (i + 1) * sf_vec_size);
  - interleaved scales: the D/sf_vec_size scale bytes of one token stay
    together as one 32-bit word; word slot k of the block's scale region
    holds token (k % W) * (bs / W) + k // W, W = 4 (the page's formula with
    its _SF_PER_INT32 = 4 bytes per int32).
"""
from __future__ import annotations

import math

import numpy as np

SF_PER_WORD = 4  # UE8M0 bytes per int32 word


def e2m1_value(code: int) -> float:
    """FP4 E2M1: 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit;
    exponent field 0 is subnormal (0 or 0.5); no infinities, no NaN."""
    code &= 0xF
    sign = -1.0 if code & 0x8 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        v = m * 0.5
    else:
        v = (1.0 + m / 2.0) * 2.0 ** (e - 1)
    return sign * v


def e2m1_table() -> np.ndarray:
    return np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)


def ue8m0_value(byte: int) -> float:
    """UE8M0 scale: 2^(byte - 127); the byte 0xFF encodes NaN."""
    byte &= 0xFF
    return math.nan if byte == 0xFF else math.ldexp(1.0, byte - 127)


def ue8m0_table() -> np.ndarray:
    return np.array([ue8m0_value(b) for b in range(256)], dtype=np.float64)


def decode_fp4_row(packed: np.ndarray, scale_bytes: np.ndarray, sf_vec: int) -> np.ndarray:
    """Values of one row: packed [D/2] uint8 (value 2i in the low nibble of
    byte i), scale_bytes [D/sf_vec] uint8 (one per sf_vec consecutive values)."""
    t = e2m1_table()
    lo = t[packed & 0xF]
    hi = t[packed >> 4]
    vals = np.empty(2 * packed.size, dtype=np.float64)
    vals[0::2] = lo
    vals[1::2] = hi
    sc = ue8m0_table()[np.asarray(scale_bytes, dtype=np.int64)]
    return vals * np.repeat(sc, sf_vec)


def required_table_columns(context_len: int, block_size: int) -> int:
    """The page's table-width precondition: round_up(L, 128) // block_size."""
    return ((context_len + 127) // 128) * 128 // block_size


def sf_slot_token(slot: int, block_size: int, interleaved: bool) -> int:
    """Token whose scale word sits at word slot `slot` of a block's scale region."""
    if not interleaved:
        return slot
    return (slot % SF_PER_WORD) * (block_size // SF_PER_WORD) + slot // SF_PER_WORD


def token_scale_bytes(block: np.ndarray, slot: int, D: int, sf_vec: int, interleaved: bool) -> np.ndarray:
    """The D/sf_vec scale bytes of token `slot` of one kv_fused block
    ([bs * (D/2 + D/sf_vec)] uint8)."""
    bs = block.size // (D // 2 + D // sf_vec)
    nsf = D // sf_vec
    data_bytes = bs * (D // 2)
    if interleaved:
        # find the word slot that holds this token
        k = next(k for k in range(bs) if sf_slot_token(k, bs, True) == slot)
    else:
        k = slot
    return block[data_bytes + k * nsf: data_bytes + (k + 1) * nsf]


def mqa_logits(w, rows=None) -> np.ndarray:
    """Logits of workload w (a workloads.Fp4Logits) as float64
    [B * next_n, max_context_len], or only the given query rows r."""
    q = _np(w.q).astype(np.uint8)
    sfq = _np(w.sf_q).astype(np.int64) & 0xFFFFFFFF
    kv = _np(w.kv_fused).astype(np.uint8).reshape(w.num_blocks, -1)
    wt = _np(w.weights).astype(np.float64)
    table = _np(w.block_table).astype(np.int64)
    lens = _np(w.context_lens).astype(np.int64)
    B, n, H, D, bs, sfv = w.B, w.n, w.H, w.D, w.bs, w.sf_vec
    nsf = D // sfv
    rows = range(B * n) if rows is None else rows
    out = np.full((len(rows), w.max_context_len), -np.inf, dtype=np.float64)
    for i, r in enumerate(rows):
        b, j = divmod(int(r), n)
        L = int(lens[b])
        vis = L - (n - 1 - j) if w.causal else L
        if vis <= 0:
            continue
        # q^ for every head of the row
        qh = np.empty((H, D), dtype=np.float64)
        for h in range(H):
            word = int(sfq[b, j, h])
            sb = np.array([(word >> (8 * s)) & 0xFF for s in range(nsf)], dtype=np.uint8)
            qh[h] = decode_fp4_row(q[b, j, h], sb, sfv)
        # k^ of every visible token, walked through the block table
        kh = np.empty((vis, D), dtype=np.float64)
        for t in range(vis):
            blk = int(table[b, t // bs])
            if blk < 0 or blk >= w.num_blocks:
                raise ValueError("oracle: block id out of range")
            block = kv[blk]
            slot = t % bs
            data = block[slot * (D // 2): (slot + 1) * (D // 2)]
            kh[t] = decode_fp4_row(data, token_scale_bytes(block, slot, D, sfv, w.sf_interleaved), sfv)
        s = qh @ kh.T                      # [H, vis] per-head dot products
        if w.rectify:
            s = np.maximum(s, 0.0)
        out[i, :vis] = wt[r] @ s          # weighted sum over heads
    return out


def _np(t):
    if t is None:
        return None
    if hasattr(t, "detach"):
        return t.detach().cpu().numpy()
    return np.asarray(t)
