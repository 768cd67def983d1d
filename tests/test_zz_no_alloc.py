"""pa_attention_noalloc: the whole attention for callers that cannot allocate
device memory, such as a plugin whose host application passes it only its
input and output buffers (no workspace argument; the library's static 32 MiB
device scratch is used instead).  Checked against pa_attention on the same
inputs, twice in a row, through the C ABI: the two run the same plan rule,
kernels and launch shape, so their results must be equal bit for bit.  This
file is collected last (see conftest), after every other test of the session
has run in the same process."""
import ctypes
import math

import pytest
import torch

import paged_attention_quantized_gb300 as pa
from paged_attention_quantized_gb300 import build as pabuild
from paged_attention_quantized_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pabuild.build()


def _ptr(t):
    return None if t is None else t.data_ptr()


def _noalloc(w, p, out, lse):
    st = pa.binding().raw_status(
        "pa_attention_noalloc", ctypes.byref(p), _ptr(w.q), _ptr(w.k_pool), _ptr(w.v_pool), _ptr(w.block_table),
        _ptr(w.context_lens), _ptr(w.k_scale), _ptr(w.v_scale), _ptr(out), _ptr(lse), pa.stream_handle())
    assert st == pa.binding().PA_OK


@pytest.fixture(scope="module", autouse=True)
def _stale_scratch(_lib):
    # a larger split problem first, so the shared scratch holds other plan
    # records and partials when the cases below run
    w = W.make("bf16", device="cuda", B=24, L_lo=500, L_hi=6000, Hq=32, Hkv=8, seed=99)
    p = pa.problem(w)
    out = torch.empty((w.B, w.n, w.Hq, w.Dv), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.B, w.n, w.Hq), dtype=torch.float32, device="cuda")
    _noalloc(w, p, out, lse)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()


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
    for _ in range(2):
        out = torch.full_like(ref, math.nan)
        lse = torch.full_like(ref_lse, math.nan)
        _noalloc(w, p, out, lse)
        torch.cuda.synchronize()
        assert torch.isfinite(out.float()).all()
        assert torch.equal(out, ref) and torch.equal(lse, ref_lse)


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
