"""GPU parity of the online softmax when the row maximum keeps growing from
page to page (K rows scaled up with their logical position), so that the
lazy running maximum is reduced and O rescaled many times within one piece,
and when it only falls (K scaled down), so that it is set once and never
moved.  Both kernel layouts: tokens on the MMA M axis (bf16 decode, 4 query
rows per kv head) and query rows on M with paired warps (E4M3 verify, D=256).
Compared with the CPU oracle on the same bytes.  Needs a GB300."""
import dataclasses

import numpy as np
import pytest
import torch

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


def _scaled_k(w, factor):
    """The workload with K row t of every request multiplied by factor(t)
    (bf16 codes scaled; E4M3 codes re-encoded from the scaled values at the
    unchanged per-tensor scale)."""
    rb = w.Dk * W.BITS[w.kv_dtype] // 8
    k = w.k_pool.clone()
    kv = k[:, : w.Hkv * w.bs * rb].view(w.num_blocks, w.Hkv, w.bs, rb)
    L = w.context_lens.cpu().tolist()
    tab = w.block_table.cpu()
    blks, slots, facs = [], [], []
    for b, Lb in enumerate(L):
        t = np.arange(Lb)
        blks.append(tab[b, t // w.bs].numpy())
        slots.append(t % w.bs)
        facs.append(np.array([factor(int(x)) for x in t], dtype=np.float32))
    blk = torch.as_tensor(np.concatenate(blks), dtype=torch.long, device=k.device)
    slot = torch.as_tensor(np.concatenate(slots), dtype=torch.long, device=k.device)
    f = torch.as_tensor(np.concatenate(facs), device=k.device)[:, None, None]
    rows = kv[blk, :, slot, :]                      # [tokens, Hkv, rb] bytes
    if w.kv_dtype == "bf16":
        x = rows.contiguous().view(torch.bfloat16).float() * f
        new = x.to(torch.bfloat16).view(torch.uint8)
    else:
        x = rows.contiguous().view(torch.float8_e4m3fn).float() * f
        new = W.e4m3_codes(x)
    kv[blk, :, slot, :] = new
    return dataclasses.replace(w, k_pool=k)


CASES = [
    ("bf16", dict(B=3, L_lo=300, L_hi=700), lambda t: 1.0 + 0.03 * t),    # grows ~20x: many rescales
    ("bf16", dict(B=3, L_lo=300, L_hi=700), lambda t: 8.0 / (1.0 + 0.03 * t)),  # only falls
    ("e4m3", dict(B=2, L_lo=200, L_hi=500), lambda t: 1.0 + 0.02 * t),
    ("e4m3", dict(B=2, L_lo=200, L_hi=500), lambda t: 6.0 / (1.0 + 0.02 * t)),
]


@pytest.mark.parametrize("name,kw,factor", CASES, ids=["bf16-grow", "bf16-fall", "e4m3-grow", "e4m3-fall"])
@pytest.mark.parametrize("split", [0, 5])
def test_growing_and_falling_scores(name, kw, factor, split):
    # With scores this peaked an output approaches single V rows (|v| up to
    # ~5), where rounding a bf16 output alone costs up to 2^-6.  E4M3: fp32
    # output (P is f16 in the kernel).  bf16 KV (P is bf16 for the bf16 MMA,
    # 2^-9 relative per weight): V scaled by 1/4, exactly, so the outputs
    # stay below 1.25 and both roundings within the bf16 bound.
    w = _scaled_k(W.make(name, device="cuda", **kw), factor)
    if name == "e4m3":
        w = dataclasses.replace(w, out_dtype="f32")
    else:
        v = (w.v_pool.view(torch.bfloat16).float() * 0.25).to(torch.bfloat16).view(torch.uint8)
        w = dataclasses.replace(w, v_pool=v.contiguous())
    out, lse, ws, _ = run_gpu(w, grid_ctas=split)
    assert error_bits(ws) == 0
    compare(w, out, lse)
