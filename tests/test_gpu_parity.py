"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle, plus
the bitwise invariances and device-side error handling.  Needs a GB300."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_attention_quantized_gb300 as pa
from paged_attention_quantized_gb300 import build as pabuild
from paged_attention_quantized_gb300 import workloads as W
from tests import notes
from tests.gpu_check import compare, error_bits, run_gpu, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pabuild.build()
    pa.binding()


def make(name, **kw):
    return W.make(name, device="cuda", **kw)


# ------------------------------------------------------------ small parity

SMALL = [
    ("tiny", dict(), 0),
    ("tiny", dict(), 1),
    ("bf16", dict(B=5, L_lo=1, L_hi=700, Hq=8, Hkv=2), 0),
    ("bf16", dict(B=5, L_lo=1, L_hi=700, Hq=8, Hkv=2), 3),
    ("bf16", dict(B=3, L_lo=100, L_hi=300, Hq=64, Hkv=2), 2),   # 32 rows: two row blocks
    ("bf16", dict(B=4, L_lo=1, L_hi=40, Hq=2, Hkv=2, n=3), 1),  # causal, n=3
    ("e4m3", dict(B=4, L_lo=4, L_hi=900, Hq=16, Hkv=4), 0),
    ("e4m3", dict(B=4, L_lo=4, L_hi=900, Hq=16, Hkv=4), 2),
    ("e4m3", dict(B=3, L_lo=1, L_hi=70, Hq=4, Hkv=1, n=4), 1),
    ("e4m3", dict(B=4, L_lo=4, L_hi=900, Hq=16, Hkv=2), 3),     # tensor-core kernel, 32 rows (two groups of 16)
    ("e4m3", dict(B=3, L_lo=4, L_hi=700, Hq=24, Hkv=2), 0),     # 48 rows (two groups of 24)
    ("e4m3", dict(B=3, L_lo=4, L_hi=700, Hq=16, Hkv=1, bs=16), 4),  # 64 rows (four groups of 16), 16-token blocks
    ("int8", dict(B=4, L_lo=1, L_hi=600, Hq=16, Hkv=2), 0),
    ("int8", dict(B=4, L_lo=1, L_hi=600, Hq=16, Hkv=2), 2),
    ("int4", dict(B=4, L_lo=1, L_hi=600, Hq=16, Hkv=2), 0),
    ("int4", dict(B=4, L_lo=1, L_hi=600, Hq=16, Hkv=2), 3),
]


@pytest.mark.parametrize("name,kw,split", SMALL, ids=lambda x: str(x))  # split: persistent CTAs (0 = default)
def test_small_parity(name, kw, split):
    w = make(name, **kw)
    out, lse, ws, _ = run_gpu(w, grid_ctas=split)
    assert error_bits(ws) == 0
    compare(w, out, lse)


@pytest.mark.parametrize("name", ["int8", "int4"])
def test_quantized_channel_scales_soft_softmax(name):
    # q scaled down (scores of order 1) so the softmax mixes many tokens:
    # checks the dequant and the fold with the plain relative tolerance
    w = make(name, B=4, L_lo=20, L_hi=500, Hq=16, Hkv=2)
    w.q = (w.q.float() / 1e7).to(w.q.dtype)
    out, lse, ws, _ = run_gpu(w, grid_ctas=2)
    compare(w, out, lse)


@pytest.mark.parametrize("name,D", [("tiny", 128), ("tiny", 256), ("bf16", 64), ("e4m3", 64), ("e4m3", 128),
                                    ("int8", 64), ("int8", 256), ("int4", 256)])
def test_other_head_dims(name, D):
    w = make(name, B=3, L_lo=1, L_hi=300, Hq=8, Hkv=2, D=D)
    out, lse, ws, _ = run_gpu(w, grid_ctas=2)
    assert error_bits(ws) == 0
    compare(w, out, lse)


@pytest.mark.parametrize("name,kw", [
    ("bf16", dict(D=256)),                 # 4 channel segments, 2 per warp
    ("int8", dict(D=256)),                 # 2 segments, 1 per warp
    ("e4m3", dict()),                      # the verify recipe's shape
    ("f16", dict(D=256)),
])
@pytest.mark.parametrize("split", [0, 3])
def test_paired_warps_d256(name, kw, split):
    # D = 256 with 16 query rows per kv head: two warps share a ring and split
    # the channel segments (scores summed through shared memory)
    base = "tiny" if name == "f16" else name
    w = make(base, B=4, L_lo=1, L_hi=600, Hq=8, Hkv=2, n=4, **kw)
    p = pa.problem(w, grid_ctas=split)
    lo = pa.binding().pa_workspace_layout(p)
    if name == "e4m3":  # E4M3 at D = 256 with 16 rows runs on the tensor-core kernel instead
        assert lo.rows_per_segment == 16 and lo.work_page_tokens == 128 and lo.warps == lo.grid_ctas
    else:
        assert lo.warps == lo.grid_ctas * 2  # two warps per worker
    out, lse, ws, _ = run_gpu(w, grid_ctas=split)
    assert error_bits(ws) == 0
    compare(w, out, lse)
    o2, l2, _, _ = run_gpu(W.relocate(w, seed=2), grid_ctas=split)
    assert torch.equal(out, o2) and torch.equal(lse, l2)


def test_steps_separately_equal_fused_call():
    w = make("bf16", B=6, L_lo=1, L_hi=2000, Hq=8, Hkv=2)
    o1, l1, _, _ = run_gpu(w, grid_ctas=5)
    o2, l2, _, _ = run_gpu(w, grid_ctas=5, steps="plan+run+combine")
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


# --------------------------------------------------------- bitwise contracts


@pytest.mark.parametrize("name", ["bf16", "e4m3", "int8", "int4"])
def test_relocation_bitwise(name):
    w = make(name, B=6, L_lo=1, L_hi=1500, Hq=16, Hkv=2)
    out, lse, _, _ = run_gpu(w)
    for s in (11, 12):
        w2 = W.relocate(w, seed=s)
        o2, l2, _, _ = run_gpu(w2)
        assert torch.equal(out, o2) and torch.equal(lse, l2)


@pytest.mark.parametrize("name", ["bf16", "e4m3", "int8", "int4", "tiny"])
def test_poisoned_padding_bitwise_and_finite(name):
    kw = {} if name == "tiny" else dict(B=6, L_lo=1, L_hi=1500, Hq=16, Hkv=2)
    w = make(name, poison=False, **kw)
    out, lse, _, _ = run_gpu(w)
    w2 = W.poison_unreferenced(w, seed=3)
    o2, l2, ws, _ = run_gpu(w2)
    assert torch.isfinite(o2).all()
    assert torch.equal(out, o2) and torch.equal(lse, l2)
    assert error_bits(ws) == 0


def test_repeat_runs_bitwise():
    w = make("e4m3", B=5, L_lo=1, L_hi=3000, Hq=32, Hkv=8, n=4)
    o1, l1, _, _ = run_gpu(w)
    o2, l2, _, _ = run_gpu(w)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_split_counts_agree_within_tolerance():
    w = make("bf16", B=4, L_lo=500, L_hi=3000, Hq=8, Hkv=2)
    outs = [run_gpu(w, grid_ctas=s)[0].float() for s in (1, 7, 0, 3000)]
    for o in outs[1:]:
        assert (o - outs[0]).abs().max().item() <= 1e-2


# -------------------------------------------------------------------- plan


@pytest.mark.parametrize("kw", [dict(), dict(grid_ctas=3), dict(grid_ctas=50), dict(num_sms=7)])
def test_plan_matches_oracle_plan(kw):
    w = make("bf16", B=37, L_lo=0, L_hi=5000, Hq=8, Hkv=2)
    p = pa.problem(w, **kw)
    out, lse, ws = pa.alloc(w, p)
    pa.run(w, p, out, ws, lse, steps="plan")
    torch.cuda.synchronize()
    lo = pa.binding().pa_workspace_layout(p)
    pl = oracle.plan(w.context_lens.cpu().numpy(), bs=w.bs, Hkv=w.Hkv, max_context_len=w.max_context_len,
                     max_blocks_per_seq=w.max_blocks_per_seq, row_blocks=lo.row_blocks, warps=lo.warps)
    raw = ws.cpu().numpy()
    hdr = raw[lo.header_offset: lo.header_offset + 16].view(np.uint32)
    assert hdr[1] == pl["total_pages"] and hdr[0] == 0
    req = raw[lo.requests_offset: lo.requests_offset + 16 * w.B].view(np.int32).reshape(w.B, 4)
    assert np.array_equal(req[:, 0], w.context_lens.cpu().numpy())
    assert np.array_equal(req[:, 1], pl["pages"]) and np.array_equal(req[:, 2], pl["prefix"])
    assert np.array_equal(req[:, 3], pl["flags"])


@pytest.mark.parametrize("name,kw", [
    ("bf16", dict(Hq=8, Hkv=2)),                 # one row block
    ("bf16", dict(Hq=32, Hkv=2, n=2)),           # 32 rows: groups of 2 workers
    ("bf16", dict(Hq=64, Hkv=2, n=2, D=256)),    # 64 rows at D = 256: groups of 4 paired workers
    ("e4m3", dict(Hq=32, Hkv=8, n=16)),          # verify: the tensor-core kernel, 64-row segments
])
def test_partial_pieces_match_oracle_plan(name, kw):
    # with many workers every segment is cut into pieces: each piece's partial
    # lse slot is written, the rest of the slots are not touched; workers of a
    # group (one per row block) share one run of pages
    w = make(name, B=3, L_lo=200, L_hi=900, **kw)
    p = pa.problem(w, grid_ctas=40)
    out, lse, ws = pa.alloc(w, p)
    lo = pa.binding().pa_workspace_layout(p)
    S = lo.rows_per_segment
    ws_f = ws.view(torch.float32)
    ws_f[lo.partial_lse_offset // 4: lo.partial_lse_offset // 4 + lo.partial_slots * S] = float("nan")
    pa.run(w, p, out, ws, lse, steps="plan+run")
    torch.cuda.synchronize()
    assert lo.group_size == lo.row_blocks and lo.warps % lo.group_size == 0
    pl = oracle.plan(w.context_lens.cpu().numpy(), bs=lo.work_page_tokens, block_size=w.bs, Hkv=w.Hkv,
                     max_context_len=w.max_context_len, max_blocks_per_seq=w.max_blocks_per_seq,
                     row_blocks=lo.row_blocks, warps=lo.warps, group_size=lo.group_size)
    lse_parts = ws_f[lo.partial_lse_offset // 4:][: lo.partial_slots * S].view(-1, S).cpu().numpy()
    R = min(lo.rows_per_kv_head, S)
    written = set()
    for pc in pl["pieces"]:
        if not pc["complete"]:
            written.add(pc["slot"])
            assert np.isfinite(lse_parts[pc["slot"], :R]).all(), pc
    out2, lse2, _, _ = run_gpu(w, grid_ctas=40)
    compare(w, out2, lse2)
    untouched = [s for s in range(lo.partial_slots) if s not in written]
    assert np.isnan(lse_parts[untouched]).all()


def test_max_abs_scale_kernel():
    w = make("int8", B=2, L_lo=10, L_hi=50, Hq=16, Hkv=2)
    for ks in (w.k_scale, torch.zeros_like(w.k_scale), -w.k_scale * 3):
        w.k_scale = ks.contiguous()
        p = pa.problem(w)
        out, lse, ws = pa.alloc(w, p)
        pa.run(w, p, out, ws, lse, steps="plan")
        torch.cuda.synchronize()
        got = ws[12:16].cpu().view(torch.float32).item()
        assert got == oracle.max_abs_scale(ks.cpu().numpy().astype(np.float32).astype(np.float64))


# ---------------------------------------------------------- edge cases


def test_zero_length_and_short_requests():
    w = make("e4m3", Hq=8, Hkv=2, n=4, context_lens=[0, 1, 3, 4, 5, 33])
    out, lse, ws, _ = run_gpu(w)
    assert error_bits(ws) == 0
    compare(w, out, lse)
    o = out.float().cpu()
    assert torch.all(o[0] == 0) and torch.all(torch.isneginf(lse[0].cpu()))
    assert torch.all(o[1, :3] == 0) and torch.all(o[2, :1] == 0)


def test_empty_batch_is_a_no_op():
    w = make("bf16", Hq=8, Hkv=2, context_lens=[5])
    p = pa.problem(w)
    p.batch = 0
    out, lse, ws = pa.alloc(w, p)
    pa.run(w, p, out, ws, lse)
    torch.cuda.synchronize()
    assert torch.isnan(out).all()  # untouched


def test_worked_fold_case_on_gpu():
    # q = 100 and k_scale = 1000 with every K code zero (onnxruntime PR #32520,
    # worked case): scores are all 0, output = mean of the values, finite
    for kv in ("int8", "int4"):
        w = make(kv, B=2, Hq=16, Hkv=2, context_lens=[7, 300])
        w.q = torch.full_like(w.q, 100.0)
        w.k_scale = torch.full_like(w.k_scale, 1000.0)
        w.k_pool = torch.zeros_like(w.k_pool)
        out, lse, ws, _ = run_gpu(w, grid_ctas=4)
        assert torch.isfinite(out).all()
        compare(w, out, lse)
        assert np.allclose(lse.cpu().numpy()[:, 0, :], np.log([[7.0], [300.0]]), atol=1e-4)


def test_large_bf16_query_into_f16_mma():
    # bf16 queries far outside the f16 range (E4M3 cache -> f16 MMA): the
    # per-row power-of-two scaling keeps them exact enough
    w = make("e4m3", B=3, L_lo=10, L_hi=200, Hq=8, Hkv=2)
    w.q = (w.q.float() * 1e30).to(torch.bfloat16)
    w.softmax_scale = 1e-30 / 16
    out, lse, ws, _ = run_gpu(w)
    compare(w, out, lse)


# ----------------------------------------------------- device-side errors


def test_bad_block_id_sets_error_and_nan_fills_only_that_request():
    w = make("bf16", B=3, Hq=8, Hkv=2, context_lens=[40, 100, 70])
    w.block_table = w.block_table.clone()
    w.block_table[1, 2] = w.num_blocks + 3   # out of range, visible position
    out, lse, ws, _ = run_gpu(w)
    assert error_bits(ws) & pa.binding().PA_DEV_ERR_BLOCK_ID
    o = out.float().cpu()
    assert torch.isnan(o[1]).all()
    assert torch.isfinite(o[0]).all() and torch.isfinite(o[2]).all()
    w.block_table[1, 2] = 0                  # the null block is not a real page either
    out, lse, ws, _ = run_gpu(w)
    assert error_bits(ws) & pa.binding().PA_DEV_ERR_BLOCK_ID


def test_context_len_over_max_sets_error():
    w = make("bf16", B=3, Hq=8, Hkv=2, context_lens=[40, 100, 70])
    out, lse, ws, _ = run_gpu(w, max_context_len=80)
    assert error_bits(ws) & pa.binding().PA_DEV_ERR_CONTEXT_LEN
    o = out.float().cpu()
    assert torch.isnan(o[1]).all() and torch.isfinite(o[0]).all() and torch.isfinite(o[2]).all()


def test_stale_plan_detected():
    w = make("bf16", B=3, Hq=8, Hkv=2, context_lens=[40, 100, 70])
    p = pa.problem(w)
    out, lse, ws = pa.alloc(w, p)
    pa.run(w, p, out, ws, lse, steps="plan")
    w.context_lens[1] = 64                   # lengths change after planning
    pa.run(w, p, out, ws, lse, steps="run+combine")
    torch.cuda.synchronize()
    assert error_bits(ws) & pa.binding().PA_DEV_ERR_STALE_PLAN
    assert torch.isnan(out[1].float()).all() and torch.isfinite(out[0].float()).all()
    # a fresh plan clears the error word
    pa.run(w, p, out, ws, lse)
    torch.cuda.synchronize()
    assert error_bits(ws) == 0
    compare(w, out, lse)


# ------------------------------------------------------------ CUDA graphs


def test_graph_capture_and_replay_with_new_lengths():
    w = make("bf16", B=8, L_lo=100, L_hi=3000, Hq=8, Hkv=2)
    p = pa.problem(w, max_context_len=4000)
    out, lse, ws = pa.alloc(w, p)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        pa.run(w, p, out, ws, lse, stream=s)   # warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pa.run(w, p, out, ws, lse, stream=s)
    # new lengths within each request's allocated pages
    old = w.context_lens.cpu()
    new = (torch.rand(w.B) * old.float()).floor().to(torch.int32) + 1
    w.context_lens.copy_(new)
    out.fill_(math.nan)
    g.replay()
    torch.cuda.synchronize()
    assert error_bits(ws) == 0
    compare(w, out, lse)


# ---------------------------------------------------- full-size workloads


@pytest.mark.parametrize("name", ["bf16", "e4m3", "int8", "int4"])
def test_full_size_sampled_parity(name):
    """The benchmark's workloads at full size, in the benchmark's launch
    configuration, checked on sampled rows (including the longest request)."""
    w = make(name)
    out, lse, ws, _ = run_gpu(w)
    assert error_bits(ws) == 0
    assert torch.isfinite(out.float()).all()
    rows = sample_rows(w, 160 if name != "e4m3" else 96)
    host = oracle.HostArrays(w)
    rep = {}
    compare(w, out, lse, rows=rows, host=host, report=rep)
    notes.add(f"full-size {name}: {rep['rows']} sampled rows, max abs err {rep['max_err']:.3g}, "
              f"{rep['hull_rows']} accepted through the near-tie hull ({rep['tie_rows']} with an exact top-two "
              f"gap below 2 eps)")
    # a near tie needs two tokens within the fold's error of the maximum:
    # most rows are decided by the normwise bound
    assert rep["hull_rows"] <= rep["rows"] // 4
    # allocation invariance at full size
    w2 = W.relocate(w, seed=5)
    o2, l2, _, _ = run_gpu(w2)
    assert torch.equal(out, o2) and torch.equal(lse, l2)


# ------------------------------------------------------- blocks as work pages

LARGE_BLOCKS = [
    ("bf16", dict(D=128, bs=128, Hq=8, Hkv=2)),           # tokens on M, 16-token work pages
    ("bf16", dict(D=256, bs=64, Hq=8, Hkv=2, n=4)),       # paired warps
    ("tiny", dict(D=256, bs=48, Hq=4, Hkv=2)),            # f16, a block in three parts
    ("e4m3", dict(bs=128, Hq=8, Hkv=2)),                  # the verify shape (n=4, D=256)
    ("int8", dict(D=256, bs=96, Hq=16, Hkv=2)),
    ("int4", dict(bs=64, Hq=64, Hkv=2)),                  # 32 rows per kv head: two row blocks
]


@pytest.mark.parametrize("name,kw", LARGE_BLOCKS, ids=lambda x: str(x))
@pytest.mark.parametrize("split", [0, 5])
def test_large_blocks_as_work_pages(name, kw, split):
    """Blocks whose K and V tiles do not fit twice per worker are handled as
    equal parts of at least 16 tokens: same results as the oracle, the plan
    in those work pages, bitwise stable under relocation."""
    w = make(name, B=3, L_lo=1, L_hi=700, **kw)
    p = pa.problem(w, grid_ctas=split)
    lo = pa.binding().pa_workspace_layout(p)
    wp = lo.work_page_tokens
    assert 16 <= wp <= w.bs and w.bs % wp == 0 and wp % 16 == 0
    if name in ("bf16", "tiny"):
        assert wp < w.bs  # these shapes only fit as parts of a block
    out, lse, ws, _ = run_gpu(w, grid_ctas=split)
    assert error_bits(ws) == 0
    compare(w, out, lse)
    raw = ws.cpu().numpy()
    pl = oracle.plan(w.context_lens.cpu().numpy(), bs=wp, Hkv=w.Hkv, max_context_len=w.max_context_len,
                     max_blocks_per_seq=w.max_blocks_per_seq * (w.bs // wp), row_blocks=lo.row_blocks,
                     warps=lo.warps)
    req = raw[lo.requests_offset: lo.requests_offset + 16 * w.B].view(np.int32).reshape(w.B, 4)
    assert np.array_equal(req[:, 1], pl["pages"]) and np.array_equal(req[:, 2], pl["prefix"])
    o2, l2, _, _ = run_gpu(W.relocate(w, seed=3), grid_ctas=split)
    assert torch.equal(out, o2) and torch.equal(lse, l2)
    o3, l3, ws3, _ = run_gpu(W.poison_unreferenced(w, seed=4), grid_ctas=split)
    assert error_bits(ws3) == 0 and torch.equal(out, o3) and torch.equal(lse, l3)


# ------------------------------------------------- merged small blocks

MERGED = [
    ("int4", dict(bs=16, Hq=16, Hkv=2)),                # tokens on M, 1 KB tiles two to a page
    ("int4", dict(bs=16, Hq=64, Hkv=2)),                # 32 rows: rows on M, two row blocks
    ("int8", dict(bs=16, D=64, Hq=8, Hkv=1)),
    ("e4m3", dict(bs=16, D=64, Hq=8, Hkv=2, n=4)),      # causal verify, 16 rows
]


@pytest.mark.parametrize("name,kw", MERGED, ids=lambda x: str(x))
@pytest.mark.parametrize("split", [0, 5])
def test_merged_blocks_as_work_pages(name, kw, split):
    """16-token blocks of short rows run two to a work page: lengths of an odd
    number of blocks leave the last page half empty (its second block is not
    copied, nor its table entry read); same results as the oracle, the plan in
    32-token pages, bitwise stable under relocation and with every unused table
    entry, padding slot and unreferenced block poisoned."""
    w = make(name, B=6, L_lo=1, L_hi=700, context_lens=[1, 16, 17, 33, 48, 650], **kw)
    p = pa.problem(w, grid_ctas=split)
    lo = pa.binding().pa_workspace_layout(p)
    assert w.bs == 16 and lo.work_page_tokens == 32
    out, lse, ws, _ = run_gpu(w, grid_ctas=split)
    assert error_bits(ws) == 0
    compare(w, out, lse)
    raw = ws.cpu().numpy()
    pl = oracle.plan(w.context_lens.cpu().numpy(), bs=32, block_size=16, Hkv=w.Hkv,
                     max_context_len=w.max_context_len, max_blocks_per_seq=w.max_blocks_per_seq,
                     row_blocks=lo.row_blocks, warps=lo.warps)
    req = raw[lo.requests_offset: lo.requests_offset + 16 * w.B].view(np.int32).reshape(w.B, 4)
    assert np.array_equal(req[:, 1], pl["pages"]) and np.array_equal(req[:, 2], pl["prefix"])
    assert np.array_equal(req[:, 3], pl["flags"])
    o2, l2, _, _ = run_gpu(W.relocate(w, seed=3), grid_ctas=split)
    assert torch.equal(out, o2) and torch.equal(lse, l2)
    o3, l3, ws3, _ = run_gpu(W.poison_unreferenced(w, seed=4), grid_ctas=split)
    assert error_bits(ws3) == 0 and torch.equal(out, o3) and torch.equal(lse, l3)


def test_merged_page_bad_second_block():
    """An invalid id in the second block of a merged work page flags the error
    and NaN-fills that request only."""
    w = make("int4", B=3, bs=16, Hq=16, Hkv=2, context_lens=[40, 100, 70])
    assert pa.binding().pa_workspace_layout(pa.problem(w)).work_page_tokens == 32
    w.block_table = w.block_table.clone()
    w.block_table[1, 3] = w.num_blocks + 3   # block 3 = second half of work page 1
    out, lse, ws, _ = run_gpu(w)
    assert error_bits(ws) & pa.binding().PA_DEV_ERR_BLOCK_ID
    o = out.float().cpu()
    assert torch.isnan(o[1]).all()
    assert torch.isfinite(o[0]).all() and torch.isfinite(o[2]).all()


def test_merged_table_limit_counts_blocks():
    """With merged pages the plan still counts the table row in blocks: a
    request one token longer than its 7-block row is flagged and NaN-filled
    although its four 32-token pages would fit ceil(7 / 2) = 4, and the others
    are exact."""
    w = make("int4", B=3, bs=16, Hq=16, Hkv=2, context_lens=[40, 112, 70])
    assert w.max_blocks_per_seq == 7
    assert pa.binding().pa_workspace_layout(pa.problem(w)).work_page_tokens == 32
    ref_out, ref_lse, _, _ = run_gpu(w)
    w.context_lens = w.context_lens.clone()
    w.context_lens[1] = 113
    out, lse, ws, _ = run_gpu(w, max_context_len=200)
    assert error_bits(ws) & pa.binding().PA_DEV_ERR_CONTEXT_LEN
    o = out.float().cpu()
    assert torch.isnan(o[1]).all()
    assert torch.equal(out[0], ref_out[0]) and torch.equal(out[2], ref_out[2])


@pytest.mark.parametrize("name,kw", [
    ("bf16", dict(Hq=128, Hkv=2, n=4)),    # 256 query rows per kv head: 16 row blocks
    ("int8", dict(Hq=64, Hkv=1, n=8)),     # 512 rows, one kv head
    ("e4m3", dict(Hq=32, Hkv=4, n=16)),    # causal verify with 16 new tokens per request
])
def test_many_query_rows_per_kv_head(name, kw):
    w = make(name, B=3, L_lo=16, L_hi=400, **kw)
    lo = pa.binding().pa_workspace_layout(pa.problem(w))
    assert lo.row_blocks == lo.rows_per_kv_head // 16
    for split in (0, 7):
        out, lse, ws, _ = run_gpu(w, grid_ctas=split)
        assert error_bits(ws) == 0
        compare(w, out, lse)
