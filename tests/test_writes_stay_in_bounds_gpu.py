"""Guard bytes: every buffer a kernel writes (attention output, lse and
workspace; the insert's pools; the sparse path's output, lse and workspace)
is a window inside a larger allocation whose margins hold a fixed byte
pattern.  After each call the margins must be unchanged, and the results
must equal those of unguarded buffers bit for bit.  Needs a GB300."""
from dataclasses import replace

import pytest
import torch

import paged_attention_quantized_gb300 as pa
from paged_attention_quantized_gb300 import build as pabuild
from paged_attention_quantized_gb300 import workloads as W

pytestmark = pytest.mark.gpu

GUARD = 4096          # margin bytes on each side (a multiple of 256: windows keep their alignment)
PATTERN = 0xA5
DEVICE = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pabuild.build()
    pa.binding()


class Guarded:
    """A tensor of `shape` / `dtype` inside a pattern-filled allocation."""

    def __init__(self, shape, dtype, device=None, init=None):
        n = 1
        for s in shape:
            n *= int(s)
        self.nbytes = n * torch.empty((), dtype=dtype).element_size()
        self.raw = torch.full((2 * GUARD + self.nbytes,), PATTERN, dtype=torch.uint8, device=device or DEVICE)
        self.t = self.raw[GUARD:GUARD + self.nbytes].view(dtype).view(*shape)
        if init is not None:
            self.t.copy_(init)

    def intact(self) -> bool:
        head = self.raw[:GUARD]
        tail = self.raw[GUARD + self.nbytes:]
        return bool((head == PATTERN).all().item()) and bool((tail == PATTERN).all().item())


def _attention_case(w, grid_ctas):
    p = pa.problem(w, grid_ctas=grid_ctas)
    out, lse, ws = pa.alloc(w, p, device=DEVICE)
    pa.run(w, p, out, ws, lse)
    g_out = Guarded(out.shape, out.dtype)
    g_lse = Guarded(lse.shape, lse.dtype)
    g_ws = Guarded(ws.shape, ws.dtype, init=torch.zeros_like(ws))
    pa.run(w, p, g_out.t, g_ws.t, g_lse.t)
    torch.cuda.synchronize()
    return (out, lse), (g_out, g_lse, g_ws)


@pytest.mark.parametrize("name,kw,grid", [
    ("tiny", dict(), 1),
    ("bf16", dict(B=3, L_lo=20, L_hi=700, Hq=8, Hkv=2), 2),          # split segments: partials + combine
    ("e4m3", dict(B=2, L_lo=20, L_hi=600, Hq=16, Hkv=4), 3),         # paired warps, causal verify
    ("int8", dict(B=2, L_lo=20, L_hi=500, Hq=16, Hkv=2), 2),
    ("int4", dict(B=2, L_lo=20, L_hi=500, Hq=16, Hkv=2), 0),
    ("latent", dict(B=2, L_lo=30, L_hi=300, Hq=32), 3),
])
def test_attention_writes_stay_in_bounds(name, kw, grid):
    w = W.make(name, device=DEVICE, **kw)
    (out, lse), guarded = _attention_case(w, grid)
    assert all(g.intact() for g in guarded)
    g_out, g_lse, _ = guarded
    assert torch.equal(g_out.t.view(torch.uint8), out.view(torch.uint8))
    assert torch.equal(g_lse.t.view(torch.uint8), lse.view(torch.uint8))


@pytest.mark.parametrize("name,kw", [
    ("bf16", dict(B=3, L_lo=40, L_hi=400, Hq=8, Hkv=2, n=5)),
    ("int4", dict(B=3, L_lo=40, L_hi=400, Hq=8, Hkv=2, n=3)),
    ("latent", dict(B=2, L_lo=70, L_hi=400, Hq=16, n=3)),
])
def test_insert_writes_stay_in_bounds(name, kw):
    w = W.make(name, device=DEVICE, **kw)
    kn, vn = W.new_kv_rows(w, "bf16", seed=2)
    plain = replace(w, k_pool=w.k_pool.clone(), v_pool=None if w.v_pool is None else w.v_pool.clone())
    pa.insert(plain, pa.problem(plain), kn, vn)
    gk = Guarded(w.k_pool.shape, w.k_pool.dtype, init=w.k_pool)
    gv = None if w.v_pool is None else Guarded(w.v_pool.shape, w.v_pool.dtype, init=w.v_pool)
    wg = replace(w, k_pool=gk.t, v_pool=None if gv is None else gv.t)
    pa.insert(wg, pa.problem(wg), kn, vn)
    torch.cuda.synchronize()
    assert gk.intact() and (gv is None or gv.intact())
    assert torch.equal(gk.t, plain.k_pool)
    if gv is not None:
        assert torch.equal(gv.t, plain.v_pool)


def test_sparse_writes_stay_in_bounds():
    w = W.make("e4m3", device=DEVICE, B=2, L_lo=40, L_hi=500, Hq=16, Hkv=2, n=2)
    sel = W.make_selection(w, k=40, seed=4)
    p = pa.problem(w)
    nb = max(256, pa.binding().pa_sparse_workspace_size(p, 40))
    shape = (w.B, w.n, w.Hq, w.Dv)
    out = torch.empty(shape, dtype=torch.bfloat16, device=DEVICE)
    lse = torch.empty(shape[:3], dtype=torch.float32, device=DEVICE)
    ws = torch.zeros(nb, dtype=torch.uint8, device=DEVICE)
    pa.sparse_run(w, p, sel, out, ws, lse)
    g_out = Guarded(shape, torch.bfloat16)
    g_lse = Guarded(shape[:3], torch.float32)
    g_ws = Guarded((nb,), torch.uint8, init=torch.zeros(nb, dtype=torch.uint8, device=DEVICE))
    pa.sparse_run(w, p, sel, g_out.t, g_ws.t, g_lse.t)
    torch.cuda.synchronize()
    assert g_out.intact() and g_lse.intact() and g_ws.intact()
    assert torch.equal(g_out.t.view(torch.uint8), out.view(torch.uint8))
    assert torch.equal(g_lse.t.view(torch.uint8), lse.view(torch.uint8))
