"""GPU parity of the single-latent MQA kernel (E4M3 latent plane of 576
channels, V = its first 512, a per-token fp32 scale in every block, 64-token
pages, 64 query rows per segment, one CTA per SM) against the CPU oracle,
plus its bitwise invariances and device-side error handling.  Needs a GB300."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import paged_attention_quantized_gb300 as pa
from paged_attention_quantized_gb300 import build as pabuild
from paged_attention_quantized_gb300 import workloads as W
from tests.gpu_check import compare, error_bits, run_gpu, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pabuild.build()
    pa.binding()


def make(**kw):
    return W.make("latent", device="cuda", **kw)


SMALL = [
    (dict(B=3, L_lo=1, L_hi=300), 0),            # 256 rows per request: four row blocks
    (dict(B=3, L_lo=1, L_hi=300), 1),            # one CTA: every segment whole
    (dict(B=3, L_lo=1, L_hi=300), 5),            # segments cut between CTAs
    (dict(B=4, L_lo=60, L_hi=700, Hq=16), 3),    # 32 rows: one partly filled row block
    (dict(B=2, L_lo=1, L_hi=130, Hq=8, n=1), 0),  # decode, 8 rows
    (dict(B=2, L_lo=300, L_hi=900, Hq=40, n=3), 7),  # causal n = 3, 120 rows
]


@pytest.mark.parametrize("kw,split", SMALL, ids=lambda x: str(x))
def test_small_parity(kw, split):
    w = make(**kw)
    out, lse, ws, _ = run_gpu(w, grid_ctas=split)
    assert error_bits(ws) == 0
    compare(w, out, lse)


@pytest.mark.parametrize("out_dtype", ["f32", "f16"])
def test_output_dtypes(out_dtype):
    w = dataclasses.replace(make(B=3, L_lo=1, L_hi=400, Hq=32), out_dtype=out_dtype)
    out, lse, ws, _ = run_gpu(w, grid_ctas=4)
    assert error_bits(ws) == 0
    compare(w, out, lse)


def test_token_scales_spread_across_pages():
    # neighbouring pages' scales differ by up to 2^12: the per-page exponent of
    # P' changes from page to page and O is rescaled by the difference
    w = make(B=3, L_lo=200, L_hi=1500, Hq=16, token_scale_spread=12)
    for split in (0, 1, 6):
        out, lse, ws, _ = run_gpu(w, grid_ctas=split)
        assert error_bits(ws) == 0
        compare(w, out, lse)


def test_fp16_queries():
    w = make(B=2, L_lo=30, L_hi=300, Hq=16)
    w = dataclasses.replace(w, q=w.q.to(torch.float16), q_dtype="f16")
    out, lse, ws, _ = run_gpu(w, grid_ctas=3)
    assert error_bits(ws) == 0
    compare(w, out, lse)


def test_zero_length_and_short_requests():
    # L = 0: no page; L = 1 < n: row 0 sees nothing, row 1 one token
    w = make(context_lens=[0, 1, 2, 65, 64], Hq=16)
    out, lse, ws, _ = run_gpu(w, grid_ctas=3)
    assert error_bits(ws) == 0
    compare(w, out, lse)
    o = out.float()
    assert (o[0] == 0).all() and torch.isinf(lse[0]).all()
    assert (o[1, 0] == 0).all() and torch.isinf(lse[1, 0]).all()


def test_relocation_bitwise():
    w = make(B=4, L_lo=1, L_hi=900, Hq=32)
    for split in (0, 5):
        o1, l1, _, _ = run_gpu(w, grid_ctas=split)
        o2, l2, _, _ = run_gpu(W.relocate(w, seed=11), grid_ctas=split)
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_poisoned_padding_bitwise_and_finite():
    w = make(B=4, L_lo=1, L_hi=900, Hq=32)
    o1, l1, _, _ = run_gpu(w, grid_ctas=5)
    w2 = W.poison_unreferenced(w, seed=4)
    o2, l2, ws, _ = run_gpu(w2, grid_ctas=5)
    assert error_bits(ws) == 0
    assert torch.isfinite(o2.float()).all()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_repeat_runs_bitwise():
    w = make(B=5, L_lo=1, L_hi=2000, Hq=64)
    o1, l1, _, _ = run_gpu(w)
    o2, l2, _, _ = run_gpu(w)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_split_counts_agree_within_tolerance():
    w = make(B=3, L_lo=500, L_hi=3000, Hq=16)
    outs = [run_gpu(w, grid_ctas=s)[0].float() for s in (1, 7, 0, 500)]
    for o in outs[1:]:
        assert (o - outs[0]).abs().max().item() <= 1e-2


@pytest.mark.parametrize("Hq,ctas", [(16, 11), (128, 22)])
def test_partial_pieces_match_oracle_plan(Hq, ctas):
    # 32 rows: one row block, groups of one CTA; 256 rows: groups of four
    w = make(B=3, L_lo=200, L_hi=900, Hq=Hq)
    p = pa.problem(w, grid_ctas=ctas)
    out, lse, ws = pa.alloc(w, p)
    lo = pa.binding().pa_workspace_layout(p)
    assert lo.rows_per_segment == 64 and lo.warps == lo.grid_ctas == ctas // lo.group_size * lo.group_size
    RS = lo.rows_per_segment
    ws_f = ws.view(torch.float32)
    ws_f[lo.partial_lse_offset // 4: lo.partial_lse_offset // 4 + lo.partial_slots * RS] = float("nan")
    pa.run(w, p, out, ws, lse, steps="plan+run")
    torch.cuda.synchronize()
    pl = oracle.plan(w.context_lens.cpu().numpy(), bs=w.bs, Hkv=w.Hkv, max_context_len=w.max_context_len,
                     max_blocks_per_seq=w.max_blocks_per_seq, row_blocks=lo.row_blocks, warps=lo.warps,
                     group_size=lo.group_size)
    parts = ws_f[lo.partial_lse_offset // 4:][: lo.partial_slots * RS].view(-1, RS).cpu().numpy()
    R = lo.rows_per_kv_head
    written = set()
    for pc in pl["pieces"]:
        if not pc["complete"]:
            written.add(pc["slot"])
            assert np.isfinite(parts[pc["slot"], :R]).all(), pc
    assert written, "the split should cut some segment"
    untouched = [s for s in range(lo.partial_slots) if s not in written]
    assert np.isnan(parts[untouched]).all()


def test_bad_block_id_sets_error_and_nan_fills_only_that_request():
    w = make(B=3, L_lo=100, L_hi=400, Hq=16)
    w.block_table[1, 0] = w.num_blocks + 5  # out of range at a visible position
    out, lse, ws, _ = run_gpu(w, grid_ctas=2)
    assert error_bits(ws) & 0x1
    o = out.float()
    assert torch.isnan(o[1]).all()
    ok = [0, 2]
    rows = np.array([(b, j, h) for b in ok for j in range(w.n) for h in range(w.Hq)])
    compare(w, out, lse, rows=rows)


def test_stale_plan_detected():
    w = make(B=3, L_lo=100, L_hi=400, Hq=16)
    p = pa.problem(w)
    out, lse, ws = pa.alloc(w, p)
    pa.run(w, p, out, ws, lse, steps="plan")
    w.context_lens[0] += 1
    pa.run(w, p, out, ws, lse, steps="run+combine")
    torch.cuda.synchronize()
    assert error_bits(ws) & 0x4
    assert torch.isnan(out[0].float()).all()


def test_full_size_sampled_parity():
    """The latent benchmark workload at full size, in the benchmark's launch
    configuration, on sampled rows (including the longest request)."""
    w = make()
    out, lse, ws, _ = run_gpu(w)
    assert error_bits(ws) == 0
    assert torch.isfinite(out.float()).all()
    rows = sample_rows(w, 512)
    host = oracle.HostArrays(w)
    compare(w, out, lse, rows=rows, host=host)
    w2 = W.relocate(w, seed=5)
    o2, l2, _, _ = run_gpu(w2)
    assert torch.equal(out, o2) and torch.equal(lse, l2)
