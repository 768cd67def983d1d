"""ctypes binding of libpa.so -- argument marshalling only.

Every function here has the name and argument order of its C counterpart in
include/pa.h; pointers are passed as Python ints (e.g. tensor.data_ptr()) and
the stream as a cudaStream_t handle (torch.cuda.current_stream().cuda_stream).
Status codes other than PA_OK raise PaError.  There is no fallback: if the
library is missing, importing this module fails.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libpa.so")

PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE, PA_ERR_CUDA = range(5)
PA_F32, PA_F16, PA_BF16, PA_E4M3, PA_INT8, PA_INT4 = range(6)
PA_SCALE_NONE, PA_SCALE_TENSOR, PA_SCALE_CHANNEL, PA_SCALE_TOKEN = range(4)
PA_DEV_ERR_BLOCK_ID = 0x1
PA_DEV_ERR_CONTEXT_LEN = 0x2
PA_DEV_ERR_STALE_PLAN = 0x4
PA_DEV_ERR_TIMEOUT = 0x8
PA_DEV_ERR_PLAN_OVERFLOW = 0x10

DTYPE = {"f32": PA_F32, "f16": PA_F16, "bf16": PA_BF16, "e4m3": PA_E4M3, "int8": PA_INT8, "int4": PA_INT4}
SCALE = {"none": PA_SCALE_NONE, "tensor": PA_SCALE_TENSOR, "channel": PA_SCALE_CHANNEL, "token": PA_SCALE_TOKEN}


class PaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {_status_name(status)}")


class Problem(ctypes.Structure):
    _fields_ = [(k, ctypes.c_int32) for k in (
        "batch", "next_n", "num_q_heads", "num_kv_heads", "head_dim_k", "head_dim_v", "block_size",
        "num_blocks", "max_blocks_per_seq", "max_context_len", "q_dtype", "kv_dtype", "out_dtype",
        "k_scale_mode", "v_scale_mode", "causal", "v_is_k_prefix", "num_sms", "grid_ctas")] + \
        [("softmax_scale", ctypes.c_float)]


class Layout(ctypes.Structure):
    _fields_ = [(k, ctypes.c_size_t) for k in (
        "total_bytes", "header_offset", "requests_offset", "partial_o_offset", "partial_lse_offset")] + \
        [("partial_slots", ctypes.c_int64)] + [(k, ctypes.c_int32) for k in (
            "rows_per_kv_head", "row_blocks", "num_sms", "grid_ctas", "warps", "ring_pages_per_warp",
            "rows_per_segment", "group_size", "work_page_tokens")]


class Fp4Problem(ctypes.Structure):
    _fields_ = [(k, ctypes.c_int32) for k in (
        "batch", "next_n", "num_heads", "head_dim", "sf_vec_size", "block_size", "num_blocks",
        "max_blocks_per_seq", "max_context_len", "out_dtype", "out_stride", "causal", "rectify",
        "sf_interleaved", "num_sms", "grid_ctas")]


if not os.path.exists(LIB_PATH):
    raise ImportError(f"libpa.so is not built ({LIB_PATH}); run "
                      "`python -m paged_attention_quantized_gb300.build` (nvcc, sm_103a)")

_lib = ctypes.CDLL(LIB_PATH)
_P = ctypes.POINTER
_vp = ctypes.c_void_p

_lib.pa_version.restype = ctypes.c_int
_lib.pa_version.argtypes = []
_lib.pa_status_string.restype = ctypes.c_char_p
_lib.pa_status_string.argtypes = [ctypes.c_int]
_lib.pa_workspace_size.restype = ctypes.c_int
_lib.pa_workspace_size.argtypes = [_P(Problem), _P(ctypes.c_size_t)]
_lib.pa_workspace_layout.restype = ctypes.c_int
_lib.pa_workspace_layout.argtypes = [_P(Problem), _P(Layout)]
_lib.pa_plan.restype = ctypes.c_int
_lib.pa_plan.argtypes = [_P(Problem), _vp, _vp, _vp, ctypes.c_size_t, _vp]
_lib.pa_run.restype = ctypes.c_int
_lib.pa_run.argtypes = [_P(Problem)] + [_vp] * 8 + [ctypes.c_size_t, _vp, _vp, _vp]
_lib.pa_combine.restype = ctypes.c_int
_lib.pa_combine.argtypes = [_P(Problem), _vp, _vp, ctypes.c_size_t, _vp, _vp, _vp]
_lib.pa_attention.restype = ctypes.c_int
_lib.pa_attention.argtypes = [_P(Problem)] + [_vp] * 8 + [ctypes.c_size_t, _vp, _vp, _vp]
_lib.pa_attention_noalloc.restype = ctypes.c_int
_lib.pa_attention_noalloc.argtypes = [_P(Problem)] + [_vp] * 10
_lib.pa_insert.restype = ctypes.c_int
_lib.pa_insert.argtypes = [_P(Problem), ctypes.c_int32] + [_vp] * 9 + [_vp]
_lib.pa_sparse_workspace_size.restype = ctypes.c_int
_lib.pa_sparse_workspace_size.argtypes = [_P(Problem), ctypes.c_int32, _P(ctypes.c_size_t)]
_lib.pa_sparse_attention.restype = ctypes.c_int
_lib.pa_sparse_attention.argtypes = [_P(Problem), ctypes.c_int32] + [_vp] * 9 + [ctypes.c_size_t, _vp, _vp, _vp]
_lib.pa_fp4_logits_workspace_size.restype = ctypes.c_int
_lib.pa_fp4_logits_workspace_size.argtypes = [_P(Fp4Problem), _P(ctypes.c_size_t)]
_lib.pa_fp4_logits.restype = ctypes.c_int
_lib.pa_fp4_logits.argtypes = [_P(Fp4Problem)] + [_vp] * 7 + [ctypes.c_size_t, _vp, _vp]
_lib.pa_get_error.restype = ctypes.c_int
_lib.pa_get_error.argtypes = [_vp, _P(ctypes.c_uint32), _vp]


def _status_name(s: int) -> str:
    return _lib.pa_status_string(int(s)).decode()


def _check(st: int, where: str) -> None:
    if st != PA_OK:
        raise PaError(st, where)


def pa_version() -> int:
    return _lib.pa_version()


def pa_workspace_size(p: Problem) -> int:
    n = ctypes.c_size_t()
    _check(_lib.pa_workspace_size(ctypes.byref(p), ctypes.byref(n)), "pa_workspace_size")
    return n.value


def pa_workspace_layout(p: Problem) -> Layout:
    lo = Layout()
    _check(_lib.pa_workspace_layout(ctypes.byref(p), ctypes.byref(lo)), "pa_workspace_layout")
    return lo


def pa_plan(p: Problem, context_lens: int, k_scale, workspace: int, workspace_bytes: int, stream) -> None:
    _check(_lib.pa_plan(ctypes.byref(p), context_lens, k_scale, workspace, workspace_bytes, stream), "pa_plan")


def pa_run(p: Problem, q, k_pool, v_pool, block_table, context_lens, k_scale, v_scale, workspace,
           workspace_bytes, out, lse, stream) -> None:
    _check(_lib.pa_run(ctypes.byref(p), q, k_pool, v_pool, block_table, context_lens, k_scale, v_scale,
                       workspace, workspace_bytes, out, lse, stream), "pa_run")


def pa_combine(p: Problem, v_scale, workspace, workspace_bytes, out, lse, stream) -> None:
    _check(_lib.pa_combine(ctypes.byref(p), v_scale, workspace, workspace_bytes, out, lse, stream), "pa_combine")


def pa_attention(p: Problem, q, k_pool, v_pool, block_table, context_lens, k_scale, v_scale, workspace,
                 workspace_bytes, out, lse, stream) -> None:
    _check(_lib.pa_attention(ctypes.byref(p), q, k_pool, v_pool, block_table, context_lens, k_scale, v_scale,
                             workspace, workspace_bytes, out, lse, stream), "pa_attention")


def pa_attention_noalloc(p: Problem, q, k_pool, v_pool, block_table, context_lens, k_scale, v_scale, out, lse,
                         stream) -> None:
    """pa_attention with the library's static 32 MiB device scratch instead of a
    caller workspace (for callers that cannot allocate device memory)."""
    _check(_lib.pa_attention_noalloc(ctypes.byref(p), q, k_pool, v_pool, block_table, context_lens, k_scale,
                                     v_scale, out, lse, stream), "pa_attention_noalloc")


def pa_insert(p: Problem, src_dtype: int, k_new, v_new, block_table, context_lens, k_scale, v_scale, k_pool,
              v_pool, dev_error, stream) -> None:
    _check(_lib.pa_insert(ctypes.byref(p), int(src_dtype), k_new, v_new, block_table, context_lens, k_scale,
                          v_scale, k_pool, v_pool, dev_error, stream), "pa_insert")


def pa_sparse_workspace_size(p: Problem, top_k: int) -> int:
    n = ctypes.c_size_t()
    _check(_lib.pa_sparse_workspace_size(ctypes.byref(p), int(top_k), ctypes.byref(n)), "pa_sparse_workspace_size")
    return n.value


def pa_sparse_attention(p: Problem, top_k: int, sel, q, k_pool, v_pool, block_table, context_lens, k_scale,
                        v_scale, workspace, workspace_bytes, out, lse, stream) -> None:
    _check(_lib.pa_sparse_attention(ctypes.byref(p), int(top_k), sel, q, k_pool, v_pool, block_table,
                                    context_lens, k_scale, v_scale, workspace, workspace_bytes, out, lse, stream),
           "pa_sparse_attention")


def pa_fp4_logits_workspace_size(p: Fp4Problem) -> int:
    n = ctypes.c_size_t()
    _check(_lib.pa_fp4_logits_workspace_size(ctypes.byref(p), ctypes.byref(n)), "pa_fp4_logits_workspace_size")
    return n.value


def pa_fp4_logits(p: Fp4Problem, q, sf_q, kv_fused, weights, context_lens, block_table, workspace,
                  workspace_bytes, out, stream) -> None:
    _check(_lib.pa_fp4_logits(ctypes.byref(p), q, sf_q, kv_fused, weights, context_lens, block_table, workspace,
                              workspace_bytes, out, stream), "pa_fp4_logits")


def pa_get_error(workspace: int, stream) -> int:
    bits = ctypes.c_uint32()
    _check(_lib.pa_get_error(workspace, ctypes.byref(bits), stream), "pa_get_error")
    return bits.value


def raw_status(fn: str, *args) -> int:
    """Call a C entry point and return its status code without raising."""
    f = getattr(_lib, fn)
    return f(*args)
