"""Pins for the quantized paged KV insert oracle (oracle/insert.py): each test
ties it to something other than itself -- library conversions (torch's
float8_e4m3fn, float16 and bfloat16 casts), the E4M3 format's own grid, the
pages' integer scale divisors, quantization error bounds, block-table
gathers done with tensor indexing, and relocation.  CPU only."""
import json
import os
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
from oracle import insert as OI
from paged_attention_quantized_gb300 import workloads as W
from tests.oracle_ref import decode_rows

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_cases.json")


def _int_codes(data: np.ndarray, kv: str) -> np.ndarray:
    """Signed codes of stored bytes, by numpy views and arithmetic shifts."""
    if kv == "int8":
        return data.view(np.int8).astype(np.int64)
    lo = (data.astype(np.uint8) << 4).astype(np.int8) >> 4
    hi = data.astype(np.int8) >> 4
    out = np.empty(data.shape[:-1] + (data.shape[-1] * 2,), dtype=np.int64)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


# ------------------------------------------------------------- E4M3 encoder


def test_e4m3_encode_round_trips_every_finite_code():
    t = oracle.e4m3_table()
    codes = np.array([c for c in range(256) if not np.isnan(t[c])])
    assert codes.size == 254
    # 0x80 is -0.0 in the table and must come back as 0x80
    assert np.array_equal(OI.e4m3_encode(t[codes].astype(np.float32)), codes.astype(np.uint8))


def test_e4m3_encode_matches_torch_cast():
    rng = np.random.default_rng(11)
    n = 200_000
    x = (rng.standard_normal(n) * np.exp2(rng.uniform(-16, 9, n))).astype(np.float32)
    x = np.clip(x, -448, 448)
    pos = oracle.e4m3_table()[:0x7F]
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)       # exact ties
    assert np.array_equal(mids.astype(np.float64), (pos[:-1] + pos[1:]) / 2)
    near = np.concatenate([np.nextafter(mids, np.float32(np.inf)), np.nextafter(mids, np.float32(0))])
    x = np.concatenate([x, mids, -mids, near, -near]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = OI.e4m3_encode(x)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(x[i]), int(got[i]), int(ref[i])) for i in bad[:5]]


def test_e4m3_encode_saturates_keeps_sign_and_nan():
    y = np.array([448.0, 449.0, 464.0, 480.0, 1e9, np.inf, -449.0, -np.inf, np.nan,
                  0.0, -0.0, -1e-30, 1e-30], np.float32)
    assert OI.e4m3_encode(y).tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x7F,
                                          0x00, 0x80, 0x80, 0x00]


def test_e4m3_subnormal_ties_go_to_even():
    u = 2.0 ** -9                  # smallest subnormal step of E4M3
    y = np.array([u, 0.5 * u, 1.5 * u, 2.5 * u, 7.5 * u, 3 * 2.0 ** -5 / 2 * 2.0 ** -3], np.float32)
    # 7.5u sits between 0x07 (7u) and 0x08 (2^-6 = 8u): the even code is 0x08
    assert OI.e4m3_encode(y)[:5].tolist() == [0x01, 0x00, 0x02, 0x02, 0x08]


# ----------------------------------------------------------- other encoders


def test_integer_codes_round_half_even_and_clamp():
    y = np.array([2.5, 3.5, -2.5, -0.5, 0.5, 1.5, 126.5, 127.49, 200, -200, np.inf, -np.inf, np.nan, -0.0],
                 np.float32)
    assert OI.int_encode(y, 127).tolist() == [2, 4, -2, 0, 0, 2, 126, 127, 127, -127, 127, -127, 0, 0]
    assert OI.int_encode(y, 7).tolist() == [2, 4, -2, 0, 0, 2, 7, 7, 7, -7, 7, -7, 0, 0]


def test_f16_bf16_encoders_match_torch_casts():
    rng = np.random.default_rng(3)
    n = 100_000
    x = (rng.standard_normal(n) * np.exp2(rng.uniform(-30, 20, n))).astype(np.float32)
    x = np.concatenate([x, np.float32([65504, 65519.99, 65520, 1e30, -1e30, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -25,
                                       np.inf, -np.inf, 0.0, -0.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -9])])
    x = x.astype(np.float32)
    t = torch.from_numpy(x)
    assert np.array_equal(OI.f16_encode(x), t.to(torch.float16).view(torch.int16).numpy().view(np.uint16))
    assert np.array_equal(OI.bf16_encode(x), t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
    nan = OI.bf16_encode(np.float32([np.nan]))
    assert torch.from_numpy(nan.view(np.int16)).view(torch.bfloat16).isnan().all()


def test_source_values_decoded_exactly():
    x = torch.randn(4096) * 3
    for dt in (torch.float32, torch.float16, torch.bfloat16):
        v = x.to(dt)
        assert np.array_equal(OI.to_f32(v), v.to(torch.float32).numpy())


# ------------------------------------------------------ scales and bounds


def test_integer_scale_span_golden():
    g = json.load(open(GOLDEN))["integer_scale_span"]
    rng = np.random.default_rng(7)
    x = (rng.standard_normal((64, 128)) * np.exp2(rng.uniform(-8, 8, (1, 128)))).astype(np.float32)
    scales = {}
    for kv, div in (("int8", g["int8_divisor"]), ("int4", g["int4_divisor"])):
        s = (np.abs(x).max(axis=0) / np.float32(div)).astype(np.float32)
        scales[kv] = s
        data, tok = OI.quantize_rows(x, kv, "channel", s)
        assert tok is None and data.shape == (64, 128 * (8 if kv == "int8" else 4) // 8)
        c = _int_codes(data, kv)
        assert np.abs(c).max() == div
        # the largest magnitude of each channel lands on +-divisor
        top = np.abs(x).argmax(axis=0)
        assert np.all(np.abs(c[top, np.arange(128)]) == div)
        # round to nearest: half a step of error (plus the fp32 quotient's rounding)
        err = np.abs(x.astype(np.float64) - c * s.astype(np.float64))
        assert np.all(err <= s * (0.5 + 2.0 ** -16))
    ratio = scales["int4"] / scales["int8"]
    assert np.allclose(ratio, 127 / 7, rtol=1e-6) and round(127 / 7) == g["ratio_stated"]


def test_token_scale_closed_form():
    rng = np.random.default_rng(9)
    x = (rng.standard_normal((40, 576)) * np.exp2(rng.uniform(-12, 12, (40, 1)))).astype(np.float32)
    x[5] = 0.0
    data, s = OI.quantize_rows(x, "e4m3", "token")
    m = np.abs(x).max(axis=1)
    expect = np.where(m == 0, np.float32(1), (m / np.float32(448)).astype(np.float32))
    assert np.array_equal(s, expect.astype(np.float32))
    assert np.all(data[5] == 0)
    dec = torch.from_numpy(data).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    top = np.abs(x).argmax(axis=1)
    live = m > 0
    assert np.all(np.abs(dec[np.arange(40), top][live]) == 448.0)
    # E4M3 keeps 3 mantissa bits: relative error 2^-4 in the normal range,
    # half the subnormal step (2^-10 of the scale) below it
    y = np.abs(x.astype(np.float64) / s[:, None].astype(np.float64))
    err = np.abs(x - dec * s[:, None])
    bound = np.where(y >= 2.0 ** -6, np.abs(x) * 2.0 ** -4, s[:, None] * 2.0 ** -10) * (1 + 2.0 ** -12)
    assert np.all(err <= bound)


# ---------------------------------------------------------- the paged walk


CASES = [
    ("tiny", dict(n=3), "f16"),
    ("bf16", dict(B=3, L_lo=5, L_hi=70, Hq=4, Hkv=2, n=2), "f32"),
    ("e4m3", dict(B=3, L_lo=5, L_hi=90, Hq=4, Hkv=2, n=4), "bf16"),
    ("int8", dict(B=3, L_lo=3, L_hi=50, Hq=4, Hkv=2, n=5), "f16"),
    ("int4", dict(B=3, L_lo=17, L_hi=50, Hq=4, Hkv=2, n=17), "bf16"),
    ("latent", dict(B=2, L_lo=3, L_hi=150, Hq=4, n=3), "bf16"),
]


def _gathered(w, pool, D, which, L, n):
    """Dequantized rows at positions L_b - n .. L_b - 1, gathered with tensor
    indexing from decode_rows (library views): [B, n, Hkv, D]."""
    vals = decode_rows(w, pool, D, which)
    tab = w.block_table.cpu().to(torch.int64)
    out = torch.zeros((w.B, n, w.Hkv, D), dtype=torch.float64)
    for b, Lb in enumerate(L):
        t = torch.arange(Lb - n, Lb)
        out[b] = vals[tab[b, t // w.bs], :, t % w.bs]
    return out.numpy()


def _bound(w, x, which):
    """Per-element error bound of one quantization of x [B, n, Hkv, D]."""
    mode = w.k_scale_mode if which == "k" else w.v_scale_mode
    scale = w.k_scale if which == "k" else w.v_scale
    ax = np.abs(x)
    if w.kv_dtype == "f16":
        return np.maximum(ax * 2.0 ** -11, 2.0 ** -25)
    if w.kv_dtype == "bf16":
        return np.maximum(ax * 2.0 ** -8, 2.0 ** -134)
    if w.kv_dtype == "e4m3" and mode == "tensor":
        s = float(scale[0])
        y = ax / s
        return np.where(y > 464, ax, np.where(y >= 2.0 ** -6, ax * 2.0 ** -4, s * 2.0 ** -10)) * 1.0001
    if w.kv_dtype == "e4m3" and mode == "token":
        m = ax.max(axis=-1, keepdims=True)
        s = np.where(m == 0, 1.0, m / 448)
        return np.where(ax / s >= 2.0 ** -6, ax * 2.0 ** -4, s * 2.0 ** -10) * 1.0001
    lim = 127 if w.kv_dtype == "int8" else 7
    s = scale.cpu().double().numpy().reshape(1, 1, w.Hkv, -1)
    clamped = ax / s > lim + 0.5
    return np.where(clamped, ax, s * (0.5 + 2.0 ** -16))


@pytest.mark.parametrize("name,kw,src", CASES, ids=lambda x: str(x))
def test_insert_walks_the_table_and_writes_only_new_slots(name, kw, src):
    w = W.make(name, **kw)
    kn, vn = W.new_kv_rows(w, src, seed=4)
    kp, vp, flags = OI.insert(w, kn, vn)
    assert flags == 0
    L = w.context_lens.tolist()
    n = w.n
    w2 = replace(w, k_pool=torch.from_numpy(kp), v_pool=None if vp is None else torch.from_numpy(vp))
    for which, new, D in (("k", kn, w.Dk), ("v", vn, w.Dv)):
        if new is None:
            continue
        pool = w2.k_pool if which == "k" else w2.v_pool
        got = _gathered(w2, pool, D, which, L, n)
        x = new.to(torch.float64).numpy()
        big = np.abs(x) > 0
        assert np.all(np.abs(got - x) <= _bound(w, x, which)), which
        assert big.mean() > 0.5
        if w.kv_dtype == "f16" and src == "f16":
            assert np.array_equal(got, x)
    # every byte that no new token maps to is unchanged
    mask_k = np.zeros_like(kp, dtype=bool)
    rowk = w.k_row_bytes
    codes = w.Hkv * w.bs * rowk
    tab = w.block_table.numpy()
    for b, Lb in enumerate(L):
        for pos in range(Lb - n, Lb):
            blk, slot = tab[b, pos // w.bs], pos % w.bs
            for g in range(w.Hkv):
                mask_k[blk, (g * w.bs + slot) * rowk:(g * w.bs + slot + 1) * rowk] = True
                if w.k_scale_mode == "token":
                    mask_k[blk, codes + (g * w.bs + slot) * 4: codes + (g * w.bs + slot + 1) * 4] = True
    k0 = w.k_pool.numpy()
    assert np.array_equal(kp[~mask_k], k0[~mask_k])
    assert not np.array_equal(kp[mask_k], k0[mask_k])
    if vp is not None:
        v0 = w.v_pool.numpy()
        mask_v = mask_k if w.v_row_bytes == rowk else None
        if mask_v is not None:
            assert np.array_equal(vp[~mask_v], v0[~mask_v])


@pytest.mark.parametrize("name", ["e4m3", "int4", "latent"])
def test_insert_commutes_with_relocation(name):
    w = W.make(name, B=3, L_lo=20, L_hi=120, Hq=4, Hkv=1 if name == "latent" else 2, n=3)
    kn, vn = W.new_kv_rows(w, "bf16", seed=8)
    kp, vp, _ = OI.insert(w, kn, vn)
    after = replace(w, k_pool=torch.from_numpy(kp), v_pool=None if vp is None else torch.from_numpy(vp))
    moved_after = W.relocate(after, seed=2)
    kp2, vp2, _ = OI.insert(W.relocate(w, seed=2), kn, vn)
    assert np.array_equal(kp2, moved_after.k_pool.numpy())
    if vp is not None:
        assert np.array_equal(vp2, moved_after.v_pool.numpy())


def test_insert_then_attention_sees_the_new_tokens():
    # f16 cache, f16 rows: the inserted tokens are exact; the oracle attention
    # over the updated pool equals dense attention over old + new rows
    w = W.make("tiny", n=2)
    w.causal = True
    kn, vn = W.new_kv_rows(w, "f16", seed=6)
    kp, vp, _ = OI.insert(w, kn, vn)
    w2 = replace(w, k_pool=torch.from_numpy(kp), v_pool=torch.from_numpy(vp))
    out, _ = oracle.attention(w2, threads=2)
    out = out.reshape(w.B, w.n, w.Hq, w.Dv)
    K = decode_rows(w, w.k_pool, w.Dk, "k")
    V = decode_rows(w, w.v_pool, w.Dv, "v")
    tab = w.block_table.to(torch.int64)
    for b, Lb in enumerate(w.context_lens.tolist()):
        t = torch.arange(Lb - w.n)
        Kb = torch.cat([K[tab[b, t // w.bs], 0, t % w.bs], kn[b, :, 0].double()])
        Vb = torch.cat([V[tab[b, t // w.bs], 0, t % w.bs], vn[b, :, 0].double()])
        for j in range(w.n):
            vis = Lb - w.n + 1 + j
            for h in range(w.Hq):
                s = (Kb[:vis] @ w.q[b, j, h].double()) * w.softmax_scale
                p = torch.softmax(s, 0)
                ref = (p[:, None] * Vb[:vis]).sum(0).numpy()
                assert np.max(np.abs(out[b, j, h] - ref)) <= 1e-12


def test_insert_contract_flags():
    # request 2's two new tokens straddle a block boundary (positions 31, 32)
    w = W.make("int8", context_lens=[40, 30, 33], Hq=4, Hkv=2, n=2)
    lens = w.context_lens.clone()
    lens[1] = 1                                  # fewer tokens than new rows
    table = w.block_table.clone()
    L2 = int(lens[2])
    table[2, (L2 - 1) // w.bs] = w.num_blocks    # last new token of request 2: bad id
    w = replace(w, context_lens=lens, block_table=table)
    kn, vn = W.new_kv_rows(w, "f16", seed=1)
    kp, vp, flags = OI.insert(w, kn, vn)
    assert flags == OI.ERR_BLOCK_ID | OI.ERR_CONTEXT_LEN
    k0 = w.k_pool.numpy()
    rowk = w.k_row_bytes
    changed = {int(bk) for bk in np.nonzero((kp != k0).any(axis=1))[0]}
    tab = table.numpy()
    expect = set()
    L0 = int(lens[0])
    for pos in range(L0 - 2, L0):
        expect.add(int(tab[0, pos // w.bs]))
    expect.add(int(tab[2, (L2 - 2) // w.bs]))
    assert changed == expect
    # request 2's first new token is written, its second is not
    blk = tab[2, (L2 - 2) // w.bs]
    slot = (L2 - 2) % w.bs
    assert not np.array_equal(kp[blk, slot * rowk:(slot + 1) * rowk], k0[blk, slot * rowk:(slot + 1) * rowk])
    # a longer context than the table allows is flagged as well
    w3 = replace(w, context_lens=torch.tensor([w.max_blocks_per_seq * w.bs + 1, 5, 5], dtype=torch.int32),
                 max_context_len=10 ** 6)
    _, _, f3 = OI.insert(w3, kn, vn)
    assert f3 & OI.ERR_CONTEXT_LEN
