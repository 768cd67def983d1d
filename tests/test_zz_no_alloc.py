"""pa_attention_noalloc: the whole attention for callers that cannot allocate
device memory (no workspace argument; the library's static 32 MiB device
scratch is used instead).  Checked against pa_attention on the same inputs,
twice in a row, through the C ABI.  This file is collected last."""
import ctypes
import math

import numpy as np
import pytest
import torch

import paged_attention_quantized_gb300 as pa
from paged_attention_quantized_gb300 import build as pabuild
from paged_attention_quantized_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = {"f32": 2e-3, "bf16": 1e-2, "f16": 1e-2}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pabuild.build()


def _ptr(t):
    return None if t is None else t.data_ptr()


@pytest.mark.parametrize("name,kw", [
    ("bf16", dict(B=6, L_lo=1, L_hi=3000, Hq=16, Hkv=4)),
    ("e4m3", dict(B=4, L_lo=3, L_hi=2000, Hq=16, Hkv=4)),
    ("int8", dict(B=4, L_lo=1, L_hi=1500, Hq=16, Hkv=2)),
])
def test_noalloc_matches_workspace_path_twice(name, kw):
    B = pa.binding()
    w = W.make(name, device="cuda", **kw)
    p = pa.problem(w)
    ref, ref_lse, ws = pa.alloc(w, p)
    pa.run(w, p, ref, ws, ref_lse)
    torch.cuda.synchronize()
    assert B.pa_get_error(ws.data_ptr(), pa.stream_handle()) == 0
    tol = TOL[w.out_dtype]
    for _ in range(2):
        out = torch.full_like(ref, math.nan)
        lse = torch.full_like(ref_lse, math.nan)
        B.pa_attention_noalloc(p, _ptr(w.q), _ptr(w.k_pool), _ptr(w.v_pool), _ptr(w.block_table),
                               _ptr(w.context_lens), _ptr(w.k_scale), _ptr(w.v_scale), _ptr(out), _ptr(lse),
                               pa.stream_handle())
        torch.cuda.synchronize()
        o, r = out.double().cpu().numpy(), ref.double().cpu().numpy()
        assert np.isfinite(o).all()
        scale = np.maximum(1.0, np.abs(r)) if w.out_dtype == "f32" and name in ("int8", "int4") else 1.0
        assert np.all(np.abs(o - r) <= tol * scale)
        assert np.allclose(lse.cpu().numpy(), ref_lse.cpu().numpy(), rtol=1e-5, atol=1e-5)


def test_noalloc_rejects_problems_beyond_its_scratch():
    B = pa.binding()
    w = W.make("bf16", device="cuda", B=2, L_lo=10, L_hi=20, Hq=8, Hkv=2)
    p = pa.problem(w)
    p.batch = 4096                       # plan + partials far beyond 32 MiB
    p.num_q_heads = 64
    p.max_context_len = 1 << 17
    p.max_blocks_per_seq = (1 << 17) // w.bs
    assert pa.workspace_bytes(p) > (32 << 20)
    st = B.raw_status("pa_attention_noalloc", ctypes.byref(p), None, None, None, None, None, None, None,
                      None, None, None)
    assert st == B.PA_ERR_WORKSPACE
