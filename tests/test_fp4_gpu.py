"""FP4 (MXFP4) paged MQA logits on the GPU (pa_fp4_logits through the C ABI)
against the CPU oracle, plus the bitwise invariances and device-side errors.
Needs a GB300."""
import dataclasses
import math

import numpy as np
import pytest
import torch

import paged_attention_quantized_gb300 as pa
from oracle import mqa_logits as M
from paged_attention_quantized_gb300 import build as pabuild
from paged_attention_quantized_gb300 import workloads as W
from tests import notes

pytestmark = pytest.mark.gpu

TOL = {"f32": 2e-3, "bf16": 1e-2, "f16": 1e-2}
TORCH = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pabuild.build()
    pa.binding()


def run(w, *, grid_ctas=0, out_stride=0, fill=math.nan):
    p = pa.fp4_problem(w, grid_ctas=grid_ctas, out_stride=out_stride)
    b = pa.binding()
    ws = torch.zeros(max(256, b.pa_fp4_logits_workspace_size(p)), dtype=torch.uint8, device="cuda")
    cols = out_stride if out_stride else w.max_context_len
    out = torch.full((w.B * w.n, cols), fill, dtype=TORCH[w.out_dtype], device="cuda")
    pa.fp4_logits(w, p, out, ws)
    torch.cuda.synchronize()
    return out, b.pa_get_error(ws.data_ptr(), pa.stream_handle())


def magnitudes(w, rows=None):
    """sum_h |w_h| * sum_d |q^_hd k^_td|: the oracle on the workload with every
    sign bit cleared (the scale of each logit, for the normwise bound)."""
    clear = lambda t: t & 0x77
    wa = dataclasses.replace(w.to("cpu"), q=clear(w.q.cpu()), weights=w.weights.cpu().abs(), rectify=False)
    kv = wa.kv_fused.clone()
    data = w.bs * (w.D // 2)
    kv[:, :data] = clear(kv[:, :data])
    wa = dataclasses.replace(wa, kv_fused=kv)
    return M.mqa_logits(wa, rows=rows)


def check(w, out, rows=None):
    """GPU logits against the oracle: same -inf / NaN pattern, finite values
    within tol * max(1, magnitude)."""
    wc = w.to("cpu")
    rows = list(range(w.B * w.n)) if rows is None else list(rows)
    ref = M.mqa_logits(wc, rows=rows)
    mag = magnitudes(w, rows=rows)
    g = out[rows, : w.max_context_len].float().cpu().numpy().astype(np.float64)
    assert np.array_equal(np.isneginf(g), np.isneginf(ref)), "masked columns differ"
    assert np.array_equal(np.isnan(g), np.isnan(ref)), "NaN columns differ"
    fin = np.isfinite(ref)
    err = np.abs(g[fin] - ref[fin])
    allow = TOL[w.out_dtype] * np.maximum(1.0, mag[fin])
    assert np.all(err <= allow), f"max err {err.max()} (worst ratio {(err / allow).max():.3g})"
    return float((err / np.maximum(1.0, mag[fin])).max(initial=0.0))


# rectify=False runs the folded-query kernel (CUDA cores, next_n <= 4), rectify=True
# (and next_n > 4) the tensor-core kernel with per-head products
SMALL = [
    dict(),                                              # bf16 out, causal, 64-token blocks, n = 2, H = 64
    dict(causal=False, out_dtype="f32"),
    dict(bs=16, sf_interleaved=True),
    dict(bs=32, n=3),
    dict(bs=128, n=1, H=16, out_dtype="f16"),
    dict(n=1, H=32, sf_interleaved=True, bs=64),
    dict(scale_lo=100, scale_hi=150, out_dtype="f32"),   # scales spread over 2^50 within rows
    dict(rectify=True, out_dtype="f32"),
    dict(rectify=True),
    dict(rectify=True, bs=16, sf_interleaved=True, causal=False),
    dict(rectify=True, bs=32, n=3),                      # 192 rows: the widest S^T
    dict(rectify=True, bs=128, n=1, H=16, out_dtype="f16"),
    dict(rectify=True, scale_lo=100, scale_hi=150, out_dtype="f32"),
    dict(n=6, H=16, out_dtype="f32"),                    # more rows than the folded kernel takes
]


@pytest.mark.parametrize("kw", SMALL, ids=lambda k: ",".join(f"{a}={b}" for a, b in k.items()) or "default")
@pytest.mark.parametrize("split", [0, 5])
def test_small_parity(kw, split):
    base = dict(B=4, L_lo=1, L_hi=700)
    base.update(kw)
    w = W.make_fp4(device="cuda", **base)
    out, bits = run(w, grid_ctas=split)
    assert bits == 0
    check(w, out)


def test_short_and_empty_requests():
    w = W.make_fp4(device="cuda", context_lens=[0, 1, 2, 127, 128, 129, 257], n=2, H=16)
    out, bits = run(w, grid_ctas=3)
    assert bits == 0
    check(w, out)
    o = out.float().cpu()
    assert torch.all(torch.isneginf(o[0:2]))            # empty request: every column -inf
    assert torch.all(torch.isneginf(o[2, :]))           # L = 1, causal row 0 sees nothing


@pytest.mark.parametrize("rectify", [False, True])
def test_relocation_and_poisoned_bytes_bitwise(rectify):
    w = W.make_fp4(device="cuda", B=5, L_lo=1, L_hi=900, H=32, rectify=rectify)
    out, _ = run(w)
    o2, bits = run(W.relocate_fp4(w, seed=4))
    assert bits == 0 and torch.equal(out, o2)
    # every byte no visible token uses: NaN scales and -6 codes
    kv = w.kv_fused.clone()
    used = torch.zeros(w.num_blocks, dtype=torch.bool)
    for b, L in enumerate(w.context_lens.tolist()):
        used[w.block_table[b, : (L + w.bs - 1) // w.bs].cpu().long()] = True
    kv[(~used).to(kv.device)] = 0xFF
    # and the unused slots of every last block
    data = w.bs * (w.D // 2)
    for b, L in enumerate(w.context_lens.tolist()):
        if L % w.bs:
            blk = int(w.block_table[b, (L - 1) // w.bs])
            kv[blk, (L % w.bs) * (w.D // 2): data] = 0xFF
            kv[blk, data + (L % w.bs) * 4:] = 0xFF
    o3, bits = run(dataclasses.replace(w, kv_fused=kv))
    assert bits == 0 and torch.equal(out, o3)


def test_output_stride_and_columns_past_max_context():
    w = W.make_fp4(device="cuda", B=3, L_lo=100, L_hi=300, H=16)
    stride = w.max_context_len + 77
    out, bits = run(w, out_stride=stride, fill=7.0)
    assert bits == 0
    check(w, out)
    assert torch.all(out[:, w.max_context_len:].float() == 7.0)


@pytest.mark.parametrize("rectify", [False, True])
def test_bad_block_id_and_over_long_request_are_nan(rectify):
    w = W.make_fp4(device="cuda", context_lens=[200, 300, 150], H=16, rectify=rectify)
    w.block_table = w.block_table.clone()
    w.block_table[1, 2] = w.num_blocks + 5
    out, bits = run(w)
    assert bits & pa.binding().PA_DEV_ERR_BLOCK_ID
    o = out.float().cpu()
    # the tokens of block 2 are NaN (the tensor-core kernel NaN-fills the whole
    # 128-token tile holding it, blocks 2 and 3); nothing outside that tile is
    assert torch.isnan(o[2:4, 128:192]).all()
    assert not torch.isnan(o[2:4, :128]).any() and not torch.isnan(o[2:4, 256:]).any()
    assert not torch.isnan(o[0:2]).any() and not torch.isnan(o[4:6]).any()
    w2 = W.make_fp4(device="cuda", context_lens=[200, 300, 150], H=16, rectify=rectify)
    p = pa.fp4_problem(w2)
    p.max_context_len = 250                                             # request 1 breaks the contract
    b = pa.binding()
    ws = torch.zeros(b.pa_fp4_logits_workspace_size(p), dtype=torch.uint8, device="cuda")
    out = torch.zeros((6, 250), dtype=torch.bfloat16, device="cuda")
    pa.fp4_logits(w2, p, out, ws)
    torch.cuda.synchronize()
    assert b.pa_get_error(ws.data_ptr(), pa.stream_handle()) & b.PA_DEV_ERR_CONTEXT_LEN
    assert torch.isnan(out[2:4].float()).all() and not torch.isnan(out[0:2].float()).any()


@pytest.mark.parametrize("rectify", [False, True])
def test_repeat_runs_bitwise(rectify):
    w = W.make_fp4(device="cuda", B=3, L_lo=500, L_hi=3000, n=2, H=64, rectify=rectify)
    o1, _ = run(w, grid_ctas=7)
    o2, _ = run(w, grid_ctas=7)
    assert torch.equal(o1, o2)


@pytest.mark.parametrize("rectify", [False, True])
def test_full_size_sampled_rows(rectify):
    """The benchmark's batch (128 requests of 4K-64K tokens, 2 query rows x 64
    heads) in its launch shape, checked on sampled rows including the
    longest request's."""
    w = W.make_fp4(device="cuda", rectify=rectify)
    out, bits = run(w)
    assert bits == 0
    L = w.context_lens.cpu().numpy()
    bmax = int(np.argmax(L))
    rng = np.random.default_rng(0)
    rows = sorted({bmax * w.n, bmax * w.n + 1} | {int(x) for x in rng.integers(0, w.B * w.n, 4)})
    worst = check(w, out, rows=rows)
    notes.add(f"fp4 logits full size (rectify={rectify}): {len(rows)} sampled rows, worst |err| / magnitude "
              f"{worst:.3g}")
