"""GPU parity of sparse (selected-token) paged attention (pa_sparse_attention
through the C ABI) against the CPU oracle (oracle/sparse.py): every cache
encoding and head dim, causal multi-row selections, bitwise invariance under
page relocation and under reordering / repeating selection entries, empty
selections and flagged block ids.  Needs a GB300."""
from dataclasses import replace

import numpy as np
import pytest
import torch

from oracle import sparse as OS
import paged_attention_quantized_gb300 as pa
from paged_attention_quantized_gb300 import build as pabuild
from paged_attention_quantized_gb300 import workloads as W
from tests.gpu_check import TOL, abs_values

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available()
    pabuild.build()


def run_sparse(w, sel, out_dtype=None):
    p = pa.problem(w, out_dtype=out_dtype)
    b = pa.binding()
    nb = b.pa_sparse_workspace_size(p, int(sel.shape[-1]))
    ws = torch.zeros(max(256, nb), dtype=torch.uint8, device="cuda")
    out = torch.full((w.B, w.n, w.Hq, w.Dv), float("nan"), dtype=pa.out_torch_dtype(out_dtype or w.out_dtype),
                     device="cuda")
    lse = torch.full((w.B, w.n, w.Hq), float("nan"), dtype=torch.float32, device="cuda")
    pa.sparse_run(w, p, sel, out, ws, lse)
    torch.cuda.synchronize()
    return out, lse, b.pa_get_error(ws.data_ptr(), pa.stream_handle())


def check(w, sel, out, lse):
    ref, rlse = OS.sparse_attention(w, sel.cpu())
    ref = ref.reshape(w.B, w.n, w.Hq, w.Dv)
    rlse = rlse.reshape(w.B, w.n, w.Hq)
    o = out.double().cpu().numpy()
    tol = TOL[w.out_dtype]
    if w.kv_dtype in ("int8", "int4"):
        # per-channel fp32 outputs up to 1e5 with cancellation between tokens:
        # normwise, against sum_t p_t |v_t| (the same criterion as the dense path)
        mag, _ = OS.sparse_attention(abs_values(w), sel.cpu())
        allow = tol * np.maximum(1.0, mag.reshape(ref.shape))
    else:
        allow = tol
    assert np.all(np.abs(o - ref) <= allow)
    l = lse.double().cpu().numpy()
    fin = np.isfinite(rlse)
    assert np.array_equal(fin, np.isfinite(l))
    assert np.all(np.abs(l[fin] - rlse[fin]) <= 1e-3 * np.maximum(1.0, np.abs(rlse[fin])))


CASES = [
    ("tiny", dict(), 16),
    ("bf16", dict(B=4, L_lo=10, L_hi=700, Hq=8, Hkv=2, n=2), 64),
    ("bf16", dict(B=3, L_lo=10, L_hi=300, Hq=16, Hkv=1, D=64), 33),
    ("e4m3", dict(B=3, L_lo=10, L_hi=900, Hq=16, Hkv=2, n=4), 100),
    ("e4m3", dict(B=3, L_lo=10, L_hi=400, Hq=12, Hkv=2, D=128, n=2), 40),
    ("int8", dict(B=3, L_lo=10, L_hi=600, Hq=16, Hkv=2), 50),
    ("int4", dict(B=3, L_lo=10, L_hi=600, Hq=16, Hkv=2), 50),
    ("int4", dict(B=2, L_lo=10, L_hi=600, Hq=16, Hkv=2, D=256), 50),
]


@pytest.mark.parametrize("name,kw,k", CASES, ids=lambda x: str(x))
def test_sparse_matches_oracle(name, kw, k):
    w = W.make(name, device="cuda", **kw)
    if name in ("int8", "int4"):
        w.q = (w.q.float() / 1e5).to(w.q.dtype)
    sel = W.make_selection(w, k=k, seed=2, shared=0.8)
    out, lse, bits = run_sparse(w, sel)
    assert bits == 0
    check(w, sel, out, lse)


@pytest.mark.parametrize("name", ["int8", "int4"])
def test_sparse_per_channel_near_one_hot(name):
    # q ~ N(0, 100^2) with per-channel scales up to 1e3, as in the INT8 / INT4
    # benchmark batch: scores of order 1e6 make each softmax nearly one-hot;
    # the sparse kernel scores in fp32 (no f16 fold), so the normwise bound
    # holds without a near-tie allowance
    w = W.make(name, device="cuda", B=3, L_lo=200, L_hi=1200, Hq=16, Hkv=2)
    sel = W.make_selection(w, k=96, seed=4, shared=0.9)
    out, lse, bits = run_sparse(w, sel)
    assert bits == 0
    check(w, sel, out, lse)


def test_sparse_relocation_and_selection_order_bitwise():
    w = W.make("e4m3", device="cuda", B=3, L_lo=50, L_hi=900, Hq=16, Hkv=2, n=2)
    sel = W.make_selection(w, k=64, seed=3)
    out, lse, _ = run_sparse(w, sel)
    o2, l2, _ = run_sparse(W.relocate(w, seed=5), sel)
    perm = sel[..., torch.randperm(64)]
    o3, l3, _ = run_sparse(w, torch.cat([perm, perm[..., :7]], dim=-1).contiguous())
    assert torch.equal(out, o2) and torch.equal(lse, l2)
    assert torch.equal(out, o3) and torch.equal(lse, l3)


def test_sparse_empty_and_flagged():
    w = W.make("bf16", device="cuda", B=3, L_lo=20, L_hi=60, Hq=8, Hkv=2)
    sel = torch.full((3, 1, 8), -1, dtype=torch.int32, device="cuda")
    sel[1, 0, :3] = torch.tensor([0, 5, 9], dtype=torch.int32)
    sel[2, 0, :2] = torch.tensor([1, 2], dtype=torch.int32)
    table = w.block_table.clone()
    table[2, 0] = w.num_blocks                      # the selected tokens of request 2 map to a bad id
    w = replace(w, block_table=table)
    out, lse, bits = run_sparse(w, sel)
    assert bits == pa.binding().PA_DEV_ERR_BLOCK_ID
    assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))
    assert torch.isnan(out[2].float()).all()
    ref, _ = OS.sparse_attention(replace(w, B=2, block_table=w.block_table[:2], context_lens=w.context_lens[:2],
                                         q=w.q[:2]), sel[:2].cpu())
    assert np.max(np.abs(out[1].double().cpu().numpy().reshape(-1, w.Dv) - ref[w.Hq:])) <= 1e-2
