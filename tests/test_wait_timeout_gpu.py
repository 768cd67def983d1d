"""Bounded waits that run out, on a GPU, with no fault: a test build of the
library (every wait gives up after 2 ms instead of 2 s; PA_FAULT_INJECT) lets
the host name, in workspace header word 4, one page whose copy the producer
withholds -- no copy and no arrive -- so every wait on that ring slot runs
out.  The call returns, PA_DEV_ERR_TIMEOUT is set, the rows that page feeds
are NaN, and every other row is NaN or bit for bit the clean result: no row
is left with stale values.  Run for the grouped, single-latent and FP4
logits kernels."""
import ctypes
import math
import time

import numpy as np
import pytest
import torch

import paged_attention_quantized_gb300 as pa
from paged_attention_quantized_gb300 import build as pabuild
from paged_attention_quantized_gb300 import workloads as W

pytestmark = pytest.mark.gpu

WITHHOLD_WORD = 4


@pytest.fixture(scope="module")
def fi():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pabuild.build()
    lib = ctypes.CDLL(pabuild.build(variant="fi"))
    b = pa.binding()
    vp = ctypes.c_void_p
    lib.pa_attention.restype = ctypes.c_int
    lib.pa_attention.argtypes = [ctypes.POINTER(b.Problem)] + [vp] * 8 + [ctypes.c_size_t, vp, vp, vp]
    lib.pa_fp4_logits.restype = ctypes.c_int
    lib.pa_fp4_logits.argtypes = [ctypes.POINTER(b.Fp4Problem)] + [vp] * 7 + [ctypes.c_size_t, vp, vp]
    return lib


def _ptr(t):
    return None if t is None else t.data_ptr()


def _attention(lib, w, p, withhold=0):
    b = pa.binding()
    n = b.pa_workspace_size(p)
    ws = torch.zeros(max(256, n), dtype=torch.uint8, device="cuda")
    ws[4 * WITHHOLD_WORD: 4 * WITHHOLD_WORD + 4] = torch.tensor([withhold], dtype=torch.int32).view(torch.uint8).cuda()
    out = torch.full((w.B, w.n, w.Hq, w.Dv), math.nan, dtype=pa.out_torch_dtype(w.out_dtype), device="cuda")
    lse = torch.full((w.B, w.n, w.Hq), math.nan, dtype=torch.float32, device="cuda")
    t0 = time.perf_counter()
    st = lib.pa_attention(ctypes.byref(p), _ptr(w.q), _ptr(w.k_pool), _ptr(w.v_pool), _ptr(w.block_table),
                          _ptr(w.context_lens), _ptr(w.k_scale), _ptr(w.v_scale), _ptr(ws), n, _ptr(out),
                          _ptr(lse), pa.stream_handle())
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert st == b.PA_OK
    bits = b.pa_get_error(ws.data_ptr(), pa.stream_handle())
    total = int(ws[4:8].view(torch.int32).item())
    return out, lse, bits, total, dt


def _owner_rows(w, total, x, wp):
    """(request, kv head) whose pages position x belongs to: positions run over
    (request, kv head, page) by the plan's prefix sums (pages of wp tokens)."""
    L = w.context_lens.cpu().numpy().astype(np.int64)
    bs = wp
    P = (L + bs - 1) // bs
    base = 0
    for b in range(w.B):
        span = int(P[b]) * w.Hkv
        if x < base + span:
            return b, (x - base) // int(P[b])
        base += span
    raise AssertionError("position outside the plan")


@pytest.mark.parametrize("name,kw,split", [
    ("bf16", dict(B=5, L_lo=200, L_hi=1500, Hq=16, Hkv=2), 0),
    ("bf16", dict(B=4, L_lo=100, L_hi=900, Hq=64, Hkv=2, n=2, D=256), 5),  # groups of 4 paired workers
    ("e4m3", dict(B=4, L_lo=100, L_hi=2000, Hq=32, Hkv=8, n=4), 7),     # the E4M3 tensor-core kernel
    ("e4m3", dict(B=3, L_lo=100, L_hi=1500, Hq=32, Hkv=8, n=16), 5),    # the same with four softmax groups
    ("latent", dict(B=3, L_lo=200, L_hi=600, Hq=32), 6),
])
def test_withheld_copy_times_out_and_leaves_no_stale_rows(fi, name, kw, split):
    w = W.make(name, device="cuda", **kw)
    p = pa.problem(w, grid_ctas=split)
    ref, ref_lse, bits, total, _ = _attention(fi, w, p)
    assert bits == 0 and torch.isfinite(ref.float()).all()
    # the clean test build equals the library itself bit for bit
    out0, lse0, ws0 = pa.alloc(w, p)
    pa.run(w, p, out0, ws0, lse0)
    torch.cuda.synchronize()
    assert torch.equal(out0, ref) and torch.equal(lse0, ref_lse)

    x = (total * w.Hkv) // 2
    out, lse, bits, _, dt = _attention(fi, w, p, withhold=x + 1)
    assert bits & pa.binding().PA_DEV_ERR_TIMEOUT
    assert dt < 10.0
    b, u = _owner_rows(w, total, x, pa.binding().pa_workspace_layout(p).work_page_tokens)
    G = w.Hq // w.Hkv
    o = out.float().cpu()
    assert torch.isnan(o[b, :, u * G:(u + 1) * G]).all()
    nan_rows = torch.isnan(o).any(dim=-1)
    assert torch.equal(nan_rows, torch.isnan(o).all(dim=-1))          # a row is all NaN or all clean
    assert torch.equal(out[~nan_rows.cuda()], ref[~nan_rows.cuda()])
    # a fresh call with the same workspace contents minus the withheld page is clean again
    out2, _, bits2, _, _ = _attention(fi, w, p)
    assert bits2 == 0 and torch.equal(out2, ref)


def test_fp4_withheld_tile_times_out(fi):
    w = W.make_fp4(device="cuda", B=4, L_lo=300, L_hi=1200, H=32, rectify=True)  # the tensor-core kernel
    p = pa.fp4_problem(w, grid_ctas=5)
    b = pa.binding()
    n = b.pa_fp4_logits_workspace_size(p)

    def call(withhold):
        ws = torch.zeros(max(256, n), dtype=torch.uint8, device="cuda")
        ws[16:20] = torch.tensor([withhold], dtype=torch.int32).view(torch.uint8).cuda()
        out = torch.full((w.B * w.n, w.max_context_len), 5.0, dtype=torch.bfloat16, device="cuda")
        t0 = time.perf_counter()
        st = fi.pa_fp4_logits(ctypes.byref(p), _ptr(w.q), _ptr(w.sf_q), _ptr(w.kv_fused), _ptr(w.weights),
                              _ptr(w.context_lens), _ptr(w.block_table), _ptr(ws), n, _ptr(out), pa.stream_handle())
        torch.cuda.synchronize()
        assert st == b.PA_OK
        return out, b.pa_get_error(ws.data_ptr(), pa.stream_handle()), int(ws[4:8].view(torch.int32).item()), \
            time.perf_counter() - t0

    ref, bits, total, _ = call(0)
    assert bits == 0
    x = total // 2
    out, bits, _, dt = call(x + 1)
    assert bits & b.PA_DEV_ERR_TIMEOUT and dt < 10.0
    # tile x: request and tile index from the plan's 128-token tiles
    L = w.context_lens.cpu().numpy()
    T = (L + 127) // 128
    r = int(np.searchsorted(np.cumsum(T), x, side="right"))
    tile = x - int(np.cumsum(T)[r - 1] if r else 0)
    o = out.float().cpu()
    assert torch.isnan(o[r * w.n:(r + 1) * w.n, tile * 128:min((tile + 1) * 128, w.max_context_len)]).all()
    nan = torch.isnan(o)
    assert torch.equal(out[~nan.cuda()], ref[~nan.cuda()])               # nothing stale: NaN or the clean value
