"""Pins for the CPU oracle: each test ties it to something other than itself
(library conversions and attention, closed forms, invariances, the pages'
worked values).  CPU only."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_attention_quantized_gb300 import workloads as W
from tests.oracle_ref import reference

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_cases.json")


def _oracle_full(w):
    out, lse = oracle.attention(w, threads=4)
    return out.reshape(w.B, w.n, w.Hq, w.Dv), lse.reshape(w.B, w.n, w.Hq)


# ------------------------------------------------------------------ decoding


def test_e4m3_table_matches_torch_float8():
    t = oracle.e4m3_table()
    ref = torch.arange(256, dtype=torch.int16).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan_codes = set(np.nonzero(np.isnan(t))[0].tolist())
    assert nan_codes == {0x7F, 0xFF}
    assert nan_codes == set(np.nonzero(np.isnan(ref))[0].tolist())
    fin = ~np.isnan(t)
    assert np.array_equal(t[fin], ref[fin])
    assert np.array_equal(np.signbit(t[fin]), np.signbit(ref[fin]))


def test_e4m3_special_points():
    t = oracle.e4m3_table()
    assert t[0x7E] == 448.0
    assert t[0x08] == 2.0 ** -6
    assert t[0x01] == 2.0 ** -9
    assert t[0x80] == 0.0 and math.copysign(1.0, t[0x80]) == -1.0
    assert t[0xFE] == -448.0


def test_e4m3_round_trip_all_finite_codes():
    t = oracle.e4m3_table()
    codes = np.array([c for c in range(256) if not np.isnan(t[c])], dtype=np.int64)
    assert codes.size == 254
    enc = W.e4m3_codes(torch.from_numpy(t[codes]).to(torch.float32)).numpy().astype(np.int64)
    assert np.array_equal(enc, codes)


def test_e4m3_nan_widens_to_fp16_nan_golden():
    g = json.load(open(GOLDEN))["e4m3_nan_codes"]
    t = oracle.e4m3_table()
    for c in g["codes"]:
        assert np.isnan(t[c])
    # widened to fp16 they stay NaN (the page quotes the canonical 0x7E00,
    # which the oracle's fp16 decoder also reads as NaN)
    f = torch.tensor(g["codes"], dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float16)
    assert torch.isnan(f).all()
    assert np.isnan(oracle.f16_value(g["fp16_bits"]))


def test_f16_bf16_decode_all_patterns():
    pats = np.arange(65536, dtype=np.uint32)
    ref16 = pats.astype(np.uint16).view(np.float16).astype(np.float64)
    refbf = torch.from_numpy(pats.astype(np.uint16).view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    for p in list(range(0, 65536, 97)) + [0x7BFF, 0x0001, 0x8001, 0x7C00, 0xFC00, 0x3C00, 0x7F80, 0x0080]:
        a, b = oracle.f16_value(p), ref16[p]
        assert (np.isnan(a) and np.isnan(b)) or a == b, hex(p)
        a, b = oracle.bf16_value(p), refbf[p]
        assert (np.isnan(a) and np.isnan(b)) or a == b, hex(p)


def test_int4_decode_all_nibbles():
    for byte in range(256):
        lo = int((np.uint8(byte) << np.uint8(4)).astype(np.int8) >> 4)
        hi = int(np.uint8(byte).astype(np.int8) >> 4)
        assert oracle.int4_value(byte, 0) == lo
        assert oracle.int4_value(byte, 1) == hi


def test_int4_pack_layout_channel_order():
    codes = torch.tensor([[-8, 7, 0, -1, 3, -3]], dtype=torch.int16)
    packed = W.pack_int4(codes)
    vals = [oracle.int4_value(int(packed[0, d // 2]), d & 1) for d in range(6)]
    assert vals == [-8, 7, 0, -1, 3, -3]


# -------------------------------------------------------- attention vs SDPA

SMALL = [
    dict(name="tiny"),
    dict(name="bf16", B=3, L_lo=1, L_hi=70, Hq=8, Hkv=2),
    dict(name="bf16", B=2, L_lo=30, L_hi=60, Hq=2, Hkv=2),
    dict(name="e4m3", B=2, L_lo=5, L_hi=90, Hq=4, Hkv=2),
    dict(name="e4m3", B=3, L_lo=4, L_hi=40, Hq=4, Hkv=1, n=4),
    dict(name="int8", B=2, L_lo=10, L_hi=40, Hq=4, Hkv=2),
    dict(name="int4", B=2, L_lo=10, L_hi=40, Hq=4, Hkv=2),
    dict(name="latent", B=2, L_lo=2, L_hi=150, Hq=4),
]


@pytest.mark.parametrize("kw", SMALL, ids=lambda k: "-".join(f"{v}" for v in k.values()))
def test_oracle_matches_sdpa(kw):
    kw = dict(kw)
    name = kw.pop("name")
    w = W.make(name, **kw)
    if name in ("int8", "int4"):
        # keep the softmax away from one-hot so the comparison is informative
        w.q = (w.q.float() / 3e4).to(w.q.dtype)
    out, lse = _oracle_full(w)
    rout, rlse = reference(w)
    scale = max(1.0, float(np.abs(rout).max()))
    assert np.max(np.abs(out - rout)) <= 1e-12 * scale
    fin = np.isfinite(rlse)
    assert np.array_equal(fin, np.isfinite(lse))
    assert np.max(np.abs(lse[fin] - rlse[fin]), initial=0.0) <= 1e-10 * max(1.0, float(np.abs(rlse[fin]).max(initial=1.0)))


def test_non_causal_multi_row_matches_sdpa():
    w = W.make("e4m3", B=2, L_lo=3, L_hi=50, Hq=4, Hkv=2, n=3)
    w.causal = False
    out, lse = _oracle_full(w)
    rout, rlse = reference(w)
    assert np.max(np.abs(out - rout)) <= 1e-12 * max(1.0, float(np.abs(rout).max()))
    # every row of a request sees the same tokens: only q differs
    w.q = w.q[:, :1].expand(-1, 3, -1, -1).contiguous()
    out, _ = _oracle_full(w)
    assert np.array_equal(out[:, 0], out[:, 2])


def test_rows_subset_equals_full():
    w = W.make("bf16", B=3, L_lo=5, L_hi=60, Hq=8, Hkv=2)
    out, lse = _oracle_full(w)
    rows = [(2, 0, 7), (0, 0, 1), (1, 0, 4)]
    o2, l2 = oracle.attention(w, rows=rows)
    for i, (b, j, h) in enumerate(rows):
        assert np.array_equal(o2[i], out[b, j, h]) and l2[i] == lse[b, j, h]


# ----------------------------------------------------------------- invariances


@pytest.mark.parametrize("name", ["bf16", "e4m3", "int4", "latent"])
def test_relocation_invariance_bitwise(name):
    w = W.make(name, B=3, L_lo=20, L_hi=120, Hq=4, Hkv=1 if name == "latent" else 2)
    out, lse = _oracle_full(w)
    for s in (1, 2):
        w2 = W.relocate(w, seed=s)
        assert not torch.equal(w2.block_table, w.block_table)
        o2, l2 = _oracle_full(w2)
        assert np.array_equal(out, o2) and np.array_equal(lse, l2)


@pytest.mark.parametrize("name", ["bf16", "e4m3", "int8", "latent"])
def test_poison_invariance_bitwise_and_finite(name):
    w = W.make(name, B=3, L_lo=20, L_hi=120, Hq=4, Hkv=1 if name == "latent" else 2, poison=False)
    out, lse = _oracle_full(w)
    w2 = W.poison_unreferenced(w, seed=5)
    o2, l2 = _oracle_full(w2)
    assert np.isfinite(o2).all()
    assert np.array_equal(out, o2) and np.array_equal(lse, l2)


def test_poison_really_holds_nan_codes():
    w = W.make("e4m3", B=2, L_lo=40, L_hi=60, Hq=4, Hkv=2)
    pool = w.k_pool.numpy()
    assert ((pool[0] == 0x7F) | (pool[0] == 0xFF)).mean() > 0.05
    ref = W.referenced_mask(w)
    assert (~ref).sum() >= 2


def test_causal_rows_equal_shorter_single_row_calls():
    n = 4
    w = W.make("e4m3", B=3, L_lo=6, L_hi=80, Hq=4, Hkv=2, n=n)
    out, lse = _oracle_full(w)
    for j in range(n):
        Lj = (w.context_lens - (n - 1 - j)).clamp(min=0)
        w1 = W.Workload(**{**w.__dict__, "n": 1, "q": w.q[:, j:j + 1].contiguous(), "context_lens": Lj})
        o1, l1 = _oracle_full(w1)
        assert np.array_equal(o1[:, 0], out[:, j]) and np.array_equal(l1[:, 0], lse[:, j])


def test_row_without_visible_tokens_is_zero():
    w = W.make("e4m3", B=2, Hq=4, Hkv=2, n=4, context_lens=[2, 9])
    out, lse = _oracle_full(w)
    # request 0 has L=2 < n: rows 0 and 1 see nothing
    assert np.all(out[0, :2] == 0.0) and np.all(np.isneginf(lse[0, :2]))
    assert np.all(np.isfinite(lse[0, 2:])) and np.all(np.isfinite(lse[1]))


# ------------------------------------------------------------------ closed forms


def _k_values(w):
    from tests.oracle_ref import decode_rows
    return decode_rows(w, w.k_pool, w.Dk, "k"), decode_rows(w, w.k_pool if w.v_is_k_prefix else w.v_pool, w.Dv, "v")


def test_single_token_context_returns_its_value():
    w = W.make("bf16", B=2, Hq=4, Hkv=2, context_lens=[1, 1])
    out, lse = _oracle_full(w)
    K, V = _k_values(w)
    for b in range(2):
        blk = int(w.block_table[b, 0])
        for h in range(4):
            g = h // 2
            assert np.array_equal(out[b, 0, h], V[blk, g, 0].numpy())
            s = float((w.q[b, 0, h].double() * K[blk, g, 0]).sum()) * w.softmax_scale
            assert abs(lse[b, 0, h] - s) <= 1e-12 * max(1, abs(s))


def test_worked_fold_case_zero_codes_gives_mean_of_values():
    g = json.load(open(GOLDEN))["fold_worked_case"]
    assert g["q"] * g["k_scale"] == g["q_times_k_scale"] == 100000.0
    for kv in ("int8", "int4"):
        w = W.make(kv, B=2, Hq=4, Hkv=2, context_lens=[7, 33])
        w.q = torch.full_like(w.q, g["q"])
        w.k_scale = torch.full_like(w.k_scale, g["k_scale"])
        w.k_pool = torch.zeros_like(w.k_pool)   # every K code is 0
        out, lse = _oracle_full(w)
        assert np.isfinite(out).all() and np.isfinite(lse).all()
        _, V = _k_values(w)
        for b, L in enumerate(w.context_lens.tolist()):
            t = np.arange(L)
            blk = w.block_table[b].numpy()[t // w.bs]
            for h in range(4):
                mean = V[blk, h // 2, t % w.bs].numpy().mean(axis=0)
                assert np.allclose(out[b, 0, h], mean, rtol=1e-12, atol=1e-12 * np.abs(mean).max())
                assert abs(lse[b, 0, h] - math.log(L)) < 1e-12


def test_equal_keys_give_mean_of_values():
    w = W.make("bf16", B=2, Hq=4, Hkv=2, context_lens=[19, 40])
    # make every K row of the referenced blocks the same bytes
    kb = w.k_pool.clone()
    row = kb[int(w.block_table[0, 0]), : w.k_row_bytes].clone()
    kb[:, :] = row.repeat(kb.shape[1] // row.numel())
    w.k_pool = kb
    out, _ = _oracle_full(w)
    _, V = _k_values(w)
    for b, L in enumerate(w.context_lens.tolist()):
        t = np.arange(L)
        blk = w.block_table[b].numpy()[t // w.bs]
        for h in range(4):
            mean = V[blk, h // 2, t % w.bs].numpy().mean(axis=0)
            assert np.allclose(out[b, 0, h], mean, rtol=1e-12, atol=1e-13)


def test_doubling_v_scale_doubles_output_exactly():
    w = W.make("int8", B=2, L_lo=10, L_hi=40, Hq=4, Hkv=2)
    out, lse = _oracle_full(w)
    w.v_scale = w.v_scale * 2.0
    o2, l2 = _oracle_full(w)
    assert np.array_equal(o2, 2.0 * out) and np.array_equal(l2, lse)


def test_scaling_q_by_power_of_two_scales_scores():
    w = W.make("bf16", B=2, L_lo=10, L_hi=40, Hq=4, Hkv=2)
    _, lse = _oracle_full(w)
    w.softmax_scale *= 0.0   # all scores 0 -> lse = ln(vis)
    _, l0 = _oracle_full(w)
    for b, L in enumerate(w.context_lens.tolist()):
        assert np.allclose(l0[b], math.log(L), rtol=0, atol=1e-12)


# --------------------------------------------------------------- merge identity


def test_lse_merge_of_token_chunks_equals_whole_row():
    w = W.make("bf16", B=2, Hq=4, Hkv=2, context_lens=[200, 77])
    out, lse = _oracle_full(w)
    for C in (1, 3, 5):
        parts_o, parts_l = [], []
        P = [(int(L) + w.bs - 1) // w.bs for L in w.context_lens.tolist()]
        S = max(-(-p // C) for p in P)
        for s in range(S):
            lens, tabs = [], []
            for b, L in enumerate(w.context_lens.tolist()):
                p0, p1 = min(s * C, P[b]), min((s + 1) * C, P[b])
                lens.append(max(0, min(L, p1 * w.bs) - p0 * w.bs))
                row = torch.zeros(w.max_blocks_per_seq, dtype=torch.int32)
                row[: p1 - p0] = w.block_table[b, p0:p1]
                tabs.append(row)
            ws = W.Workload(**{**w.__dict__, "context_lens": torch.tensor(lens, dtype=torch.int32),
                               "block_table": torch.stack(tabs)})
            o, l = _oracle_full(ws)
            parts_o.append(o)
            parts_l.append(l)
        mo, ml = oracle.lse_merge(np.stack(parts_o), np.stack(parts_l))
        assert np.allclose(mo, out, rtol=1e-12, atol=1e-13)
        assert np.allclose(ml, lse, rtol=1e-13, atol=1e-12)


def test_lse_merge_empty_chunks():
    o = np.array([[[1.0, 2.0]], [[5.0, 6.0]]])
    l = np.array([[-np.inf], [-np.inf]])
    mo, ml = oracle.lse_merge(o, l)
    assert np.all(mo == 0) and np.all(np.isneginf(ml))
    l = np.array([[-np.inf], [0.5]])
    mo, ml = oracle.lse_merge(o, l)
    assert np.array_equal(mo[0], [5.0, 6.0]) and ml[0] == 0.5


# ------------------------------------------------------------------- fold scale


def test_max_abs_scale():
    assert oracle.max_abs_scale(np.array([[0.5, -3.0], [2.0, 1.0]], dtype=np.float32)) == 3.0
    assert oracle.max_abs_scale(np.zeros((2, 4), dtype=np.float32)) == 1.0
    g = json.load(open(GOLDEN))["fold_bound"]
    ks = np.array([1e-2, 3.0, -1e3, 7.0], dtype=np.float64)
    q = 100.0
    m = oracle.max_abs_scale(ks)
    assert np.all(np.abs(q * ks / m) <= abs(q)), g["claim"]


# -------------------------------------------------------------------- near ties


def _tie_workload(codes0, n=1, causal=False, v_seed=0):
    """INT8 per-channel cache (scales 1), one kv head, D = 64, softmax scale
    1/8, q = e_0: the exact score of token t is codes0[t] / 8, so scores are
    fixed by hand (every value below is exact in binary)."""
    L = len(codes0)
    w = W.make("int8", B=1, Hq=1, Hkv=1, D=64, n=n, context_lens=[L])
    w.causal = causal
    q = torch.zeros_like(w.q, dtype=torch.float32)
    q[..., 0] = 1.0
    w.q = q.to(w.q.dtype)
    w.k_scale = torch.ones_like(w.k_scale)
    rng = np.random.default_rng(v_seed)
    w.v_scale = torch.from_numpy(rng.uniform(0.5, 2.0, size=tuple(w.v_scale.shape)).astype(np.float32))
    k = w.k_pool.clone()
    rb = w.k_row_bytes
    for t, c in enumerate(codes0):
        blk = int(w.block_table[0, t // w.bs])
        slot = t % w.bs
        row = k[blk, slot * rb:(slot + 1) * rb]
        row[0] = int(np.int8(c).view(np.uint8))
    w.k_pool = k
    assert w.softmax_scale == 0.125
    return w


def _v_values(w, tokens):
    """Decoded V rows (code * v_scale) of the given logical tokens."""
    out = []
    rb = w.v_row_bytes
    vs = w.v_scale.numpy().astype(np.float64)[0]
    for t in tokens:
        blk = int(w.block_table[0, t // w.bs])
        slot = t % w.bs
        codes = w.v_pool[blk, slot * rb:(slot + 1) * rb].numpy().view(np.int8).astype(np.float64)
        out.append(codes * vs)
    return np.array(out)


# scores (code / 8): 12.5 at token 22 (the maximum), 12.0 at 3 and 11.5 at 37
# (within 1.0), 11.0 at 17 (exactly 1.5 below), everything else <= 50 / 8
_TIE_CODES = [((t * 7) % 51) - 20 for t in range(40)]
for _t, _c in ((3, 96), (17, 88), (22, 100), (37, 92)):
    _TIE_CODES[_t] = _c


def test_row_ties_selects_exactly_within_delta_of_the_maximum():
    w = _tie_workload(_TIE_CODES)
    vmin, vmax, gap, cnt = oracle.row_ties(w, 0, 0, 0, delta=1.0)
    assert cnt == 3                                   # 12.5, 12.0, 11.5 (the bound itself is inside)
    assert gap == 0.5                                 # exact distance to the runner-up
    ref = _v_values(w, [3, 22, 37])
    assert np.array_equal(vmin, ref.min(axis=0)) and np.array_equal(vmax, ref.max(axis=0))
    vmin, vmax, gap, cnt = oracle.row_ties(w, 0, 0, 0, delta=1.5)
    assert cnt == 4
    ref = _v_values(w, [3, 17, 22, 37])
    assert np.array_equal(vmin, ref.min(axis=0)) and np.array_equal(vmax, ref.max(axis=0))
    # a delta that puts M - delta one ulp above 11.5 (the ulp of scores in
    # [8, 16) is 2^-49) drops the token at exactly M - delta; likewise at 12.0
    _, _, _, cnt = oracle.row_ties(w, 0, 0, 0, delta=1.0 - 2.0 ** -49)
    assert cnt == 2
    _, _, _, cnt = oracle.row_ties(w, 0, 0, 0, delta=0.5 - 2.0 ** -49)
    assert cnt == 1
    vmin, vmax, _, cnt = oracle.row_ties(w, 0, 0, 0, delta=0.0)
    assert cnt == 1
    ref = _v_values(w, [22])[0]
    assert np.array_equal(vmin, ref) and np.array_equal(vmax, ref)


def test_row_ties_exact_tie_and_maximum_at_the_ends():
    codes = list(_TIE_CODES)
    codes[0] = 100                                    # ties the maximum, first token
    w = _tie_workload(codes)
    vmin, vmax, gap, cnt = oracle.row_ties(w, 0, 0, 0, delta=0.0)
    assert gap == 0.0 and cnt == 2
    ref = _v_values(w, [0, 22])
    assert np.array_equal(vmin, ref.min(axis=0)) and np.array_equal(vmax, ref.max(axis=0))
    codes = list(_TIE_CODES)
    codes[39] = 104                                   # a new maximum, last token: 13.0
    w = _tie_workload(codes)
    vmin, vmax, gap, cnt = oracle.row_ties(w, 0, 0, 0, delta=1.0)
    assert gap == 0.5 and cnt == 3                    # 13.0, 12.5, 12.0
    ref = _v_values(w, [3, 22, 39])
    assert np.array_equal(vmin, ref.min(axis=0)) and np.array_equal(vmax, ref.max(axis=0))


def test_row_ties_respects_the_causal_horizon():
    codes = list(_TIE_CODES)
    codes[39] = 104                                   # visible to the last query row only
    w = _tie_workload(codes, n=2, causal=True)
    _, _, gap, cnt = oracle.row_ties(w, 0, 0, 0, delta=1.0)   # row 0 sees tokens 0..38
    assert gap == 0.5 and cnt == 3                    # 12.5, 12.0, 11.5
    _, _, gap, cnt = oracle.row_ties(w, 0, 1, 0, delta=1.0)   # row 1 sees token 39 too
    assert gap == 0.5 and cnt == 3                    # 13.0, 12.5, 12.0


def test_row_ties_single_token_and_whole_row():
    w = _tie_workload(_TIE_CODES[:1])
    vmin, vmax, gap, cnt = oracle.row_ties(w, 0, 0, 0, delta=0.0)
    assert cnt == 1 and gap == math.inf
    w = _tie_workload(_TIE_CODES)
    out, _ = _oracle_full(w)
    vmin, vmax, gap, cnt = oracle.row_ties(w, 0, 0, 0, delta=float("inf"))
    assert cnt == 40
    ref = _v_values(w, range(40))
    assert np.array_equal(vmin, ref.min(axis=0)) and np.array_equal(vmax, ref.max(axis=0))
    assert np.all(out[0, 0, 0] >= vmin - 1e-12) and np.all(out[0, 0, 0] <= vmax + 1e-12)


def test_bad_block_id_is_reported_not_read():
    w = W.make("bf16", B=2, Hq=4, Hkv=2, context_lens=[5, 17])
    w.block_table = w.block_table.clone()
    w.block_table[1, 1] = w.num_blocks + 5
    with pytest.raises(ValueError, match="block id"):
        oracle.attention(w)
