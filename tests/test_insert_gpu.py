"""GPU parity of the quantized paged KV insert (pa_insert through the C ABI)
against the CPU oracle (oracle/insert.py): byte for byte on every pool byte,
for every cache encoding and source dtype, ragged and block-crossing inserts,
relocation, contract violations, non-finite inputs, the attention over the
written pool, and sampled tokens of full-size inserts.  Needs a GB300."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
from oracle import insert as OI
import paged_attention_quantized_gb300 as pa
from paged_attention_quantized_gb300 import build as pabuild
from paged_attention_quantized_gb300 import workloads as W
from tests.gpu_check import compare, error_bits, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pabuild.build()
    pa.binding()


def gpu_insert(w, kn, vn):
    """Insert into copies of w's pools; returns (workload with the new pools,
    device error bits)."""
    w2 = replace(w, k_pool=w.k_pool.clone(), v_pool=None if w.v_pool is None else w.v_pool.clone())
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.insert(w2, pa.problem(w2), kn, vn, dev_error=err)
    torch.cuda.synchronize()
    return w2, int(err.item()) & 0xFFFFFFFF


def assert_pools_equal(w2, kp, vp):
    assert np.array_equal(w2.k_pool.cpu().numpy(), kp)
    if vp is not None:
        assert np.array_equal(w2.v_pool.cpu().numpy(), vp)


CASES = [
    # name, workload overrides, source dtype
    ("tiny", dict(n=3), "f16"),
    ("tiny", dict(n=1), "f32"),
    ("tiny", dict(n=5), "bf16"),
    ("bf16", dict(B=5, L_lo=40, L_hi=700, Hq=8, Hkv=2, n=1), "bf16"),
    ("bf16", dict(B=4, L_lo=40, L_hi=700, Hq=8, Hkv=2, n=37), "f32"),     # crosses blocks
    ("bf16", dict(B=3, L_lo=40, L_hi=300, Hq=8, Hkv=2, D=64, n=2), "f16"),
    ("bf16", dict(B=3, L_lo=40, L_hi=300, Hq=8, Hkv=2, D=256, bs=64, n=9), "bf16"),
    ("e4m3", dict(B=4, L_lo=8, L_hi=900, Hq=16, Hkv=4, n=4), "bf16"),
    ("e4m3", dict(B=4, L_lo=8, L_hi=900, Hq=16, Hkv=4, n=4), "f32"),
    ("e4m3", dict(B=3, L_lo=8, L_hi=400, Hq=8, Hkv=2, D=64, n=1), "f16"),
    ("e4m3", dict(B=3, L_lo=80, L_hi=400, Hq=8, Hkv=2, D=128, bs=128, n=70), "bf16"),
    ("int8", dict(B=4, L_lo=1, L_hi=600, Hq=16, Hkv=2, n=1), "f16"),
    ("int8", dict(B=4, L_lo=20, L_hi=600, Hq=16, Hkv=2, n=19), "f32"),
    ("int8", dict(B=3, L_lo=20, L_hi=300, Hq=8, Hkv=2, D=64, n=3), "bf16"),
    ("int8", dict(B=3, L_lo=20, L_hi=300, Hq=8, Hkv=2, D=256, bs=32, n=3), "f16"),
    ("int4", dict(B=4, L_lo=1, L_hi=600, Hq=16, Hkv=2, n=1), "f16"),
    ("int4", dict(B=4, L_lo=20, L_hi=600, Hq=16, Hkv=2, n=16), "bf16"),
    ("int4", dict(B=3, L_lo=20, L_hi=300, Hq=8, Hkv=2, D=256, n=5), "f32"),
    ("latent", dict(B=3, L_lo=2, L_hi=700, Hq=16, n=2), "bf16"),
    ("latent", dict(B=3, L_lo=70, L_hi=700, Hq=16, n=65), "f32"),        # more than a block of new tokens
    ("latent", dict(B=2, L_lo=2, L_hi=300, Hq=16, n=1), "f16"),
]


@pytest.mark.parametrize("name,kw,src", CASES, ids=lambda x: str(x))
def test_insert_matches_oracle_bytewise(name, kw, src):
    w = W.make(name, device="cuda", **kw)
    kn, vn = W.new_kv_rows(w, src, seed=21)
    w2, bits = gpu_insert(w, kn, vn)
    assert bits == 0
    kp, vp, flags = OI.insert(w, kn, vn)
    assert flags == 0
    assert_pools_equal(w2, kp, vp)


def test_insert_empty_batch_writes_nothing():
    w = W.make("int8", device="cuda", B=2, L_lo=20, L_hi=60, Hq=4, Hkv=2)
    w0 = replace(w, B=0, block_table=w.block_table[:0], context_lens=w.context_lens[:0])
    kn, vn = W.new_kv_rows(w0, "f16", seed=1)
    w2, bits = gpu_insert(w0, kn, vn)
    assert bits == 0
    assert torch.equal(w2.k_pool, w.k_pool) and torch.equal(w2.v_pool, w.v_pool)


def test_insert_twice_is_idempotent_and_repeatable():
    w = W.make("e4m3", device="cuda", B=3, L_lo=8, L_hi=400, Hq=8, Hkv=2, n=3)
    kn, vn = W.new_kv_rows(w, "bf16", seed=2)
    a, _ = gpu_insert(w, kn, vn)
    b, _ = gpu_insert(a, kn, vn)
    assert torch.equal(a.k_pool, b.k_pool) and torch.equal(a.v_pool, b.v_pool)


@pytest.mark.parametrize("name", ["bf16", "int4", "latent"])
def test_insert_commutes_with_relocation(name):
    w = W.make(name, device="cuda", B=3, L_lo=20, L_hi=300, Hq=4, Hkv=1 if name == "latent" else 2, n=3)
    kn, vn = W.new_kv_rows(w, "bf16", seed=3)
    a, _ = gpu_insert(w, kn, vn)
    moved = W.relocate(a, seed=4)
    b, _ = gpu_insert(W.relocate(w, seed=4), kn, vn)
    assert torch.equal(b.k_pool, moved.k_pool)
    if b.v_pool is not None:
        assert torch.equal(b.v_pool, moved.v_pool)


def test_insert_contract_violations_flag_and_skip():
    w = W.make("int8", device="cuda", context_lens=[40, 30, 33, 50], Hq=4, Hkv=2, n=2)
    lens = w.context_lens.clone()
    lens[1] = 1                                   # fewer tokens than new rows
    table = w.block_table.clone()
    table[2, 32 // w.bs] = w.num_blocks           # request 2's last new token: id out of range
    table[3, 49 // w.bs] = 0                      # request 3's last new token: the null block
    w = replace(w, context_lens=lens, block_table=table)
    kn, vn = W.new_kv_rows(w, "f16", seed=5)
    w2, bits = gpu_insert(w, kn, vn)
    kp, vp, flags = OI.insert(w, kn, vn)
    assert flags == OI.ERR_BLOCK_ID | OI.ERR_CONTEXT_LEN
    assert bits == flags
    assert_pools_equal(w2, kp, vp)
    # longer than max_context_len, and more pages than table columns
    for lens2, mctx in (([40, 30, 33, 50], 45), ([40, 30, 33, w.max_blocks_per_seq * w.bs + 1], 10 ** 6)):
        w3 = replace(w, block_table=w.block_table.clone(), max_context_len=mctx,
                     context_lens=torch.tensor(lens2, dtype=torch.int32, device="cuda"))
        w4, bits = gpu_insert(w3, kn, vn)
        kp, vp, flags = OI.insert(w3, kn, vn)
        assert bits == flags and flags & OI.ERR_CONTEXT_LEN
        assert_pools_equal(w4, kp, vp)


@pytest.mark.parametrize("name", ["e4m3", "int8", "int4", "latent", "bf16"])
def test_insert_non_finite_inputs(name):
    w = W.make(name, device="cuda", B=3, L_lo=20, L_hi=300, Hq=4, Hkv=1 if name == "latent" else 2, n=4)
    kn, vn = W.new_kv_rows(w, "f32", seed=6)
    kn = kn.clone()
    kn[0, 0, 0, :3] = torch.tensor([float("nan"), float("inf"), -float("inf")])
    kn[1, 2, 0, 5] = float("nan")                # one NaN in an otherwise finite row
    kn[2, 1, 0] = 0.0                            # an all-zero row
    w2, bits = gpu_insert(w, kn, vn)
    assert bits == 0
    kp, vp, _ = OI.insert(w, kn, vn)
    got = w2.k_pool.cpu().numpy()
    if w.kv_dtype == "e4m3":
        # NaN codes may carry either sign: compare NaN-ness there, bytes elsewhere
        codes = w.Hkv * w.bs * w.k_row_bytes
        gc, rc = got[:, :codes], kp[:, :codes]
        nan_ref = (rc & 0x7F) == 0x7F
        nan_got = (gc & 0x7F) == 0x7F
        assert np.array_equal(nan_ref, nan_got)
        assert np.array_equal(gc[~nan_ref], rc[~nan_ref])
        assert np.array_equal(got[:, codes:], kp[:, codes:]) or w.k_scale_mode == "token"
        if w.k_scale_mode == "token":
            # scales of NaN rows are NaN (any payload); the others match bitwise
            sg = got[:, codes:].copy().view(np.float32)
            sr = kp[:, codes:].copy().view(np.float32)
            assert np.array_equal(np.isnan(sg), np.isnan(sr))
            assert np.array_equal(sg[~np.isnan(sr)], sr[~np.isnan(sr)])
    elif w.kv_dtype == "bf16":
        # NaN payloads may differ: compare values as bf16, NaN-ness for NaNs
        g16 = torch.from_numpy(got.view(np.int16)).view(torch.bfloat16).float().numpy()
        r16 = torch.from_numpy(kp.view(np.int16)).view(torch.bfloat16).float().numpy()
        assert np.array_equal(np.isnan(g16), np.isnan(r16))
        assert np.array_equal(got.view(np.uint16)[~np.isnan(r16)], kp.view(np.uint16)[~np.isnan(r16)])
    else:
        assert np.array_equal(got, kp)
    if vp is not None:
        assert np.array_equal(w2.v_pool.cpu().numpy(), vp)


@pytest.mark.parametrize("name,kw", [
    ("bf16", dict(B=4, L_lo=20, L_hi=500, Hq=8, Hkv=2, n=1)),
    ("e4m3", dict(B=3, L_lo=20, L_hi=500, Hq=16, Hkv=4, n=4)),
    ("int8", dict(B=3, L_lo=20, L_hi=500, Hq=16, Hkv=2, n=1)),
    ("latent", dict(B=2, L_lo=20, L_hi=400, Hq=32, n=2)),
])
def test_attention_over_inserted_tokens(name, kw):
    # insert on the GPU, attend on the GPU; the oracle attends over the pool
    # the oracle's insert wrote (the same bytes, checked above)
    w = W.make(name, device="cuda", **kw)
    if name == "int8":
        w.q = (w.q.float() / 1e7).to(w.q.dtype)   # a softmax that mixes many tokens
    # rows drawn like the pool's own values: the absolute tolerance of bf16
    # outputs assumes outputs of order 1 (half a bf16 step at 8 is 0.016)
    kn, vn = W.new_kv_rows(w, "bf16", seed=7, outliers=False)
    w2, _ = gpu_insert(w, kn, vn)
    grid = dict(grid_ctas=3) if name == "latent" else {}
    out, lse, ws, _ = run_gpu(w2, **grid)
    assert error_bits(ws) == 0
    kp, vp, _ = OI.insert(w, kn, vn)
    ref_w = replace(w2, k_pool=torch.from_numpy(kp), v_pool=None if vp is None else torch.from_numpy(vp))
    ref_w = ref_w.to("cpu")
    # compare() evaluates the oracle on the workload it is given
    compare(ref_w, out, lse)


@pytest.mark.parametrize("name,n", [("int8", 128), ("latent", 64), ("bf16", 256)])
def test_full_size_insert_sampled(name, n):
    # the benchmark's insert step: 16384 new tokens into the full-size pool;
    # sampled tokens are checked byte for byte, every other byte is unchanged
    w = W.make(name, device="cuda", n=n)
    kn, vn = W.new_kv_rows(w, "bf16" if name != "int8" else "f16", seed=8)
    before_k = w.k_pool.clone()
    w2, bits = gpu_insert(w, kn, vn)
    assert bits == 0
    L = w.context_lens.cpu().numpy()
    tab = w.block_table.cpu().numpy()
    rng = np.random.default_rng(9)
    picks = {(int(np.argmax(L)), n - 1), (0, 0)}
    while len(picks) < 256:
        picks.add((int(rng.integers(w.B)), int(rng.integers(n))))
    ks = None if w.k_scale is None else w.k_scale.cpu()
    row = w.k_row_bytes
    codes = w.Hkv * w.bs * row
    mask = torch.zeros_like(w.k_pool, dtype=torch.bool)
    for b in range(w.B):
        pos = torch.arange(int(L[b]) - n, int(L[b]))
        blk = torch.as_tensor(tab[b])[pos // w.bs].to(torch.int64)
        slot = pos % w.bs
        for g in range(w.Hkv):
            start = (g * w.bs + slot) * row
            idx = start[:, None] + torch.arange(row)[None]
            mask[blk.cuda()[:, None], idx.cuda()] = True
            if w.k_scale_mode == "token":
                s0 = codes + (g * w.bs + slot) * 4
                sidx = s0[:, None] + torch.arange(4)[None]
                mask[blk.cuda()[:, None], sidx.cuda()] = True
    assert torch.equal(w2.k_pool[~mask], before_k[~mask])
    got = w2.k_pool
    for b, j in sorted(picks):
        pos = int(L[b]) - n + j
        blk, slot = int(tab[b, pos // w.bs]), pos % w.bs
        for g in range(w.Hkv):
            s = None if ks is None else (ks.reshape(-1)[:1] if w.k_scale_mode == "tensor" else ks[g])
            data, tok = OI.quantize_rows(OI.to_f32(kn[b, j, g]), w.kv_dtype, w.k_scale_mode, s)
            o = (g * w.bs + slot) * row
            assert np.array_equal(got[blk, o:o + row].cpu().numpy(), data), (b, j, g)
            if tok is not None:
                t = codes + (g * w.bs + slot) * 4
                assert np.array_equal(got[blk, t:t + 4].cpu().numpy(), np.float32(tok).reshape(1).view(np.uint8))
