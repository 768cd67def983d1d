"""Paged decode / verify attention over a quantized paged KV cache on GB300.

The computation lives in libpa.so (CUDA, sm_103a) behind the C ABI of
include/pa.h; this package is its thin Python face:

  * `_binding`  -- ctypes declarations of pa_workspace_size / pa_plan / pa_run /
                   pa_combine / pa_attention / pa_insert / pa_sparse_attention /
                   pa_fp4_logits / pa_get_error (same names);
  * `problem()` / `run()` -- marshal a batch held in torch CUDA tensors into
                   those calls (pointers, sizes, the current stream);
  * `workloads` -- seeded synthetic inputs (no attention arithmetic).

The library is loaded lazily so that `workloads` can be used without it.
"""
from __future__ import annotations

import math
from typing import Optional

__all__ = ["problem", "workspace_bytes", "run", "insert", "sparse_run", "fp4_problem", "fp4_logits",
           "stream_handle", "binding"]


def binding():
    from . import _binding
    return _binding


def problem(w, *, num_sms: int = 0, grid_ctas: int = 0,
            max_context_len: Optional[int] = None, out_dtype: Optional[str] = None):
    """pa_problem for a workload-shaped batch (see workloads.Workload)."""
    b = binding()
    return b.Problem(
        batch=w.B, next_n=w.n, num_q_heads=w.Hq, num_kv_heads=w.Hkv, head_dim_k=w.Dk, head_dim_v=w.Dv,
        block_size=w.bs, num_blocks=w.num_blocks, max_blocks_per_seq=w.max_blocks_per_seq,
        max_context_len=w.max_context_len if max_context_len is None else max_context_len,
        q_dtype=b.DTYPE[w.q_dtype], kv_dtype=b.DTYPE[w.kv_dtype],
        out_dtype=b.DTYPE[out_dtype or w.out_dtype], k_scale_mode=b.SCALE[w.k_scale_mode],
        v_scale_mode=b.SCALE[w.v_scale_mode], causal=int(bool(w.causal)),
        v_is_k_prefix=int(bool(w.v_is_k_prefix)), num_sms=num_sms, grid_ctas=grid_ctas,
        softmax_scale=float(w.softmax_scale))


def _ptr(t) -> Optional[int]:
    return None if t is None else int(t.data_ptr())


def stream_handle(stream=None) -> int:
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def workspace_bytes(p) -> int:
    return binding().pa_workspace_size(p)


def run(w, p, out, workspace, lse=None, stream=None, *, steps: str = "all") -> None:
    """Enqueue the attention for workload tensors already on the device.

    steps: "all" (pa_attention), or any of "plan", "run", "combine"
    separated by '+'.  All buffers are caller-owned torch tensors."""
    b = binding()
    s = stream_handle(stream)
    ws, wsb = _ptr(workspace), workspace.numel() * workspace.element_size()
    args_run = (_ptr(w.q), _ptr(w.k_pool), _ptr(w.v_pool), _ptr(w.block_table), _ptr(w.context_lens),
                _ptr(w.k_scale), _ptr(w.v_scale))
    if steps == "all":
        b.pa_attention(p, *args_run, ws, wsb, _ptr(out), _ptr(lse), s)
        return
    for step in steps.split("+"):
        if step == "plan":
            b.pa_plan(p, _ptr(w.context_lens), _ptr(w.k_scale), ws, wsb, s)
        elif step == "run":
            b.pa_run(p, *args_run, ws, wsb, _ptr(out), _ptr(lse), s)
        elif step == "combine":
            b.pa_combine(p, _ptr(w.v_scale), ws, wsb, _ptr(out), _ptr(lse), s)
        else:
            raise ValueError(step)


def insert(w, p, k_new, v_new=None, dev_error=None, stream=None) -> None:
    """Enqueue pa_insert: write the new rows k_new / v_new ([B, n, Hkv, D]
    torch CUDA tensors, f32 / f16 / bf16) into w's pools in place.  dev_error:
    optional int32 CUDA tensor of one element that collects the error bits."""
    b = binding()
    src = {"torch.float32": b.PA_F32, "torch.float16": b.PA_F16, "torch.bfloat16": b.PA_BF16}[str(k_new.dtype)]
    b.pa_insert(p, src, _ptr(k_new), _ptr(v_new), _ptr(w.block_table), _ptr(w.context_lens), _ptr(w.k_scale),
                _ptr(w.v_scale), _ptr(w.k_pool), _ptr(w.v_pool), _ptr(dev_error), stream_handle(stream))


def sparse_run(w, p, sel, out, workspace, lse=None, stream=None) -> None:
    """Enqueue pa_sparse_attention for workload tensors on the device; sel is
    an int32 [B, n, top_k] CUDA tensor of selected logical positions and
    workspace a uint8 tensor of pa_sparse_workspace_size bytes."""
    b = binding()
    top_k = int(sel.shape[-1])
    b.pa_sparse_attention(p, top_k, _ptr(sel), _ptr(w.q), _ptr(w.k_pool), _ptr(w.v_pool), _ptr(w.block_table),
                          _ptr(w.context_lens), _ptr(w.k_scale), _ptr(w.v_scale), _ptr(workspace),
                          workspace.numel() * workspace.element_size(), _ptr(out), _ptr(lse), stream_handle(stream))


def out_torch_dtype(name: str):
    import torch
    return {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[name]


def alloc(w, p, device="cuda"):
    """(out, lse, workspace) tensors sized for problem p (NaN-filled out)."""
    import torch
    out = torch.full((w.B, w.n, w.Hq, w.Dv), math.nan, dtype=out_torch_dtype(w.out_dtype), device=device)
    lse = torch.full((w.B, w.n, w.Hq), math.nan, dtype=torch.float32, device=device)
    nbytes = workspace_bytes(p)
    ws = torch.zeros(max(256, nbytes), dtype=torch.uint8, device=device)
    return out, lse, ws


def fp4_problem(w, *, num_sms: int = 0, grid_ctas: int = 0, out_stride: int = 0):
    """pa_fp4_problem for an FP4 MQA-logits batch (see workloads.Fp4Logits)."""
    b = binding()
    return b.Fp4Problem(batch=w.B, next_n=w.n, num_heads=w.H, head_dim=w.D, sf_vec_size=w.sf_vec, block_size=w.bs,
                        num_blocks=w.num_blocks, max_blocks_per_seq=w.max_blocks_per_seq,
                        max_context_len=w.max_context_len, out_dtype=b.DTYPE[w.out_dtype], out_stride=out_stride,
                        causal=int(bool(w.causal)), rectify=int(bool(w.rectify)),
                        sf_interleaved=int(bool(w.sf_interleaved)), num_sms=num_sms, grid_ctas=grid_ctas)


def fp4_logits(w, p, out, workspace, stream=None) -> None:
    """Enqueue pa_fp4_logits for an Fp4Logits batch on the device; out is a
    [B * next_n, >= max_context_len] tensor of the problem's output dtype
    (its row stride is taken from p.out_stride, 0 = max_context_len) and
    workspace a uint8 tensor of pa_fp4_logits_workspace_size bytes."""
    b = binding()
    b.pa_fp4_logits(p, _ptr(w.q), _ptr(w.sf_q), _ptr(w.kv_fused), _ptr(w.weights), _ptr(w.context_lens),
                    _ptr(w.block_table), _ptr(workspace), workspace.numel(), _ptr(out), stream_handle(stream))
