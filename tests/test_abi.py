"""The C-ABI library builds, loads, exports every symbol include/pa.h declares,
and rejects bad arguments on the host.  No GPU needed: nothing here launches
a kernel (every call below fails validation or only sizes the workspace)."""
import ctypes
import os
import re

import pytest

from paged_attention_quantized_gb300 import build as pabuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def B():
    pabuild.build()
    from paged_attention_quantized_gb300 import _binding
    return _binding


def declared_symbols():
    hdr = open(os.path.join(ROOT, "include", "pa.h")).read()
    return sorted(set(re.findall(r"PA_API\s+[\w\s\*]+?\b(pa_\w+)\s*\(", hdr)))


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for name in ("pa_workspace_size", "pa_plan", "pa_run", "pa_combine", "pa_get_error"):
        assert name in syms


def test_library_exports_every_declared_symbol(B):
    lib = ctypes.CDLL(B.LIB_PATH)
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_exports_nothing_undeclared(B):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l and l.split()[-1].startswith("pa_")}
    assert exported == set(declared_symbols())


def _prob(B, **kw):
    base = dict(batch=4, next_n=1, num_q_heads=32, num_kv_heads=8, head_dim_k=128, head_dim_v=128,
                block_size=16, num_blocks=1000, max_blocks_per_seq=64, max_context_len=1024,
                q_dtype=B.PA_BF16, kv_dtype=B.PA_BF16, out_dtype=B.PA_BF16, k_scale_mode=0, v_scale_mode=0,
                causal=0, v_is_k_prefix=0, num_sms=152, grid_ctas=0, softmax_scale=0.088)
    base.update(kw)
    return B.Problem(**base)


def test_workspace_size_and_layout(B):
    p = _prob(B)
    n = B.pa_workspace_size(p)
    lo = B.pa_workspace_layout(p)
    assert n == lo.total_bytes > 0
    offs = [lo.header_offset, lo.requests_offset, lo.partial_o_offset, lo.partial_lse_offset]
    assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
    assert lo.rows_per_kv_head == 4 and lo.row_blocks == 1 and lo.num_sms == 152
    assert lo.grid_ctas % 152 == 0 and lo.warps == lo.grid_ctas * 4 and lo.ring_pages_per_warp >= 2
    assert lo.partial_slots == 4 * 8 + lo.warps and lo.rows_per_segment == 16 and lo.group_size == 1
    assert lo.partial_lse_offset - lo.partial_o_offset >= lo.partial_slots * 16 * 128 * 4


def _latent(B, **kw):
    base = dict(batch=8, next_n=2, num_q_heads=128, num_kv_heads=1, head_dim_k=576, head_dim_v=512,
                block_size=64, num_blocks=2000, max_blocks_per_seq=200, max_context_len=12800,
                q_dtype=B.PA_BF16, kv_dtype=B.PA_E4M3, out_dtype=B.PA_BF16, k_scale_mode=B.PA_SCALE_TOKEN,
                v_scale_mode=B.PA_SCALE_TOKEN, causal=1, v_is_k_prefix=1, num_sms=152, softmax_scale=1 / 24)
    base.update(kw)
    return _prob(B, **base)


def test_latent_layout(B):
    lo = B.pa_workspace_layout(_latent(B))
    assert lo.rows_per_kv_head == 256 and lo.rows_per_segment == 64 and lo.row_blocks == 4
    assert lo.grid_ctas == 152 and lo.warps == 152 and lo.ring_pages_per_warp == 2 and lo.group_size == 4
    assert lo.partial_slots == (8 * 1 + 152 // 4) * 4
    # the launch is whole groups of one CTA per row block
    for want, got in ((1, 4), (5, 4), (11, 8), (150, 148)):
        assert B.pa_workspace_layout(_latent(B, grid_ctas=want)).grid_ctas == got
    assert lo.partial_lse_offset - lo.partial_o_offset >= lo.partial_slots * 64 * 512 * 4
    assert lo.total_bytes - lo.partial_lse_offset >= lo.partial_slots * 64 * 4


@pytest.mark.parametrize("kw", [dict(block_size=32), dict(head_dim_k=512), dict(head_dim_v=256),
                                dict(kv_dtype=5, head_dim_k=576), dict(k_scale_mode=1), dict(kv_dtype=1)])
def test_latent_unsupported_variants(B, kw):
    st = B.raw_status("pa_workspace_size", ctypes.byref(_latent(B, **kw)), ctypes.byref(ctypes.c_size_t()))
    assert st == B.PA_ERR_UNSUPPORTED


def test_latent_v_wider_than_k_rejected(B):
    st = B.raw_status("pa_workspace_size", ctypes.byref(_latent(B, head_dim_v=640)), ctypes.byref(ctypes.c_size_t()))
    assert st == B.PA_ERR_INVALID_ARG


def test_latent_run_needs_no_v_pool_but_checks_the_rest(B):
    p = _latent(B)
    need = B.pa_workspace_size(p)
    # q not 16-byte aligned: rejected before any launch
    st = B.raw_status("pa_run", ctypes.byref(p), 0x4008, 0x5000, None, 0x7000, 0x8000, None, None,
                      0x10000, need, 0x9000, None, None)
    assert st == B.PA_ERR_INVALID_ARG
    st = B.raw_status("pa_run", ctypes.byref(p), 0x4000, 0x5008, None, 0x7000, 0x8000, None, None,
                      0x10000, need, 0x9000, None, None)
    assert st == B.PA_ERR_INVALID_ARG


@pytest.mark.parametrize("field,value", [
    ("batch", -1), ("next_n", 0), ("num_q_heads", 30), ("num_kv_heads", 0), ("block_size", 0),
    ("num_blocks", 0), ("max_blocks_per_seq", 0), ("max_context_len", -5), ("q_dtype", 7), ("grid_ctas", -1),
    ("q_dtype", 3), ("kv_dtype", 9), ("out_dtype", 4), ("k_scale_mode", 5), ("causal", 2),
])
def test_invalid_arguments(B, field, value):
    st = B.raw_status("pa_workspace_size", ctypes.byref(_prob(B, **{field: value})), ctypes.byref(ctypes.c_size_t()))
    assert st == B.PA_ERR_INVALID_ARG


def test_nan_softmax_scale_rejected(B):
    st = B.raw_status("pa_workspace_size", ctypes.byref(_prob(B, softmax_scale=float("nan"))),
                      ctypes.byref(ctypes.c_size_t()))
    assert st == B.PA_ERR_INVALID_ARG


@pytest.mark.parametrize("kw", [dict(head_dim_k=96, head_dim_v=96), dict(head_dim_v=64),
                                dict(block_size=24), dict(kv_dtype=5, head_dim_k=64, head_dim_v=64)])
def test_unsupported_shapes(B, kw):
    st = B.raw_status("pa_workspace_size", ctypes.byref(_prob(B, **kw)), ctypes.byref(ctypes.c_size_t()))
    assert st == B.PA_ERR_UNSUPPORTED


def test_plan_overflow_refused_on_the_host(B):
    # 33000 requests x 65536 table columns could name more than 2^31 - 1 pages:
    # refused before anything is sized or launched; one column less fits
    big = dict(batch=33000, num_q_heads=1, num_kv_heads=1, head_dim_k=64, head_dim_v=64, num_blocks=2,
               max_context_len=1 << 20, max_blocks_per_seq=65536)
    st = B.raw_status("pa_workspace_size", ctypes.byref(_prob(B, **big)), ctypes.byref(ctypes.c_size_t()))
    assert st == B.PA_ERR_UNSUPPORTED
    st = B.raw_status("pa_plan", ctypes.byref(_prob(B, **big)), None, None, None, 0, None)
    assert st == B.PA_ERR_UNSUPPORTED
    ok = dict(big, max_blocks_per_seq=65072)          # 33000 x 65072 = 2147376000 < 2^31
    assert B.pa_workspace_size(_prob(B, **ok)) > 0
    # latent problems count 64-token pages the same way
    st = B.raw_status("pa_workspace_size", ctypes.byref(_latent(B, batch=1 << 20, max_blocks_per_seq=4096)),
                      ctypes.byref(ctypes.c_size_t()))
    assert st == B.PA_ERR_UNSUPPORTED


def test_bad_workspace_rejected_before_any_launch(B):
    p = _prob(B)
    need = B.pa_workspace_size(p)
    # NULL, misaligned and too-small workspaces fail on the host
    for ws, n in ((None, need), (0x1000 + 8, need), (0x1000, need - 1)):
        assert B.raw_status("pa_plan", ctypes.byref(p), 0x2000, None, ws, n, None) == B.PA_ERR_WORKSPACE
        assert B.raw_status("pa_combine", ctypes.byref(p), None, ws, n, 0x3000, None, None) == B.PA_ERR_WORKSPACE


def test_missing_pointers_rejected(B):
    p = _prob(B, k_scale_mode=B.PA_SCALE_CHANNEL, kv_dtype=B.PA_INT8)
    need = B.pa_workspace_size(p)
    # per-channel K scales without a k_scale pointer
    assert B.raw_status("pa_plan", ctypes.byref(p), 0x2000, None, 0x10000, need, None) == B.PA_ERR_INVALID_ARG
    # misaligned pool pointer
    p2 = _prob(B)
    need2 = B.pa_workspace_size(p2)
    st = B.raw_status("pa_run", ctypes.byref(p2), 0x4000, 0x5008, 0x6000, 0x7000, 0x8000, None, None,
                      0x10000, need2, 0x9000, None, None)
    assert st == B.PA_ERR_INVALID_ARG


@pytest.mark.parametrize("latent", [False, True])
def test_partial_slots_cover_oracle_pieces(B, latent):
    import numpy as np
    import oracle
    rng = np.random.default_rng(3)
    for _ in range(20):
        Bsz = int(rng.integers(1, 60))
        bs = int(rng.choice([16, 32, 64]))
        maxctx = int(rng.integers(1, 20000))
        Hkv = int(rng.choice([1, 2, 8]))
        G = int(rng.choice([1, 4, 16]))
        n = int(rng.choice([1, 2, 4]))
        mbps = -(-maxctx // bs)
        if latent:
            bs = 64
            mbps = -(-maxctx // bs)
            p = _latent(B, batch=Bsz, max_context_len=maxctx, num_kv_heads=Hkv, num_q_heads=Hkv * G * 8,
                        next_n=n, max_blocks_per_seq=mbps, num_sms=int(rng.integers(1, 200)),
                        grid_ctas=int(rng.integers(0, 50)))
        else:
            p = _prob(B, batch=Bsz, block_size=bs, max_context_len=maxctx, num_kv_heads=Hkv, num_q_heads=Hkv * G,
                      next_n=n, max_blocks_per_seq=mbps, num_sms=int(rng.integers(1, 200)),
                      grid_ctas=int(rng.integers(0, 50)))
        lo = B.pa_workspace_layout(p)
        L = rng.integers(0, maxctx + 1, Bsz)
        pl = oracle.plan(L, bs=bs, Hkv=Hkv, max_context_len=maxctx, max_blocks_per_seq=mbps,
                         row_blocks=lo.row_blocks, warps=lo.warps, group_size=lo.group_size)
        assert pl["slots"] == lo.partial_slots
        assert all(pc["slot"] < lo.partial_slots for pc in pl["pieces"])


def test_every_block_size_has_a_launch(B):
    """Every KV encoding x head dim x block size (multiples of 16 up to 128) x
    rows per kv head gets a launch: whole blocks when two per worker fit,
    else equal work pages of >= 16 tokens; 16-token blocks of rows of at most
    64 bytes are merged two to a work page when two merged pages fit; E4M3 at
    head dim 256 with 16..64 rows per kv head runs on the tensor-core kernel
    in 128-token chunks."""
    for kv in (B.PA_F16, B.PA_BF16, B.PA_E4M3, B.PA_INT8, B.PA_INT4):
        for D in (64, 128, 256):
            if kv == B.PA_INT4 and D == 64:
                continue
            for bs in range(16, 129, 16):
                for hq, n in ((8, 1), (32, 1), (64, 1), (32, 4), (128, 2), (96, 4), (32, 16)):
                    p = _prob(B, kv_dtype=kv, head_dim_k=D, head_dim_v=D, block_size=bs, num_q_heads=hq, next_n=n)
                    lo = B.pa_workspace_layout(p)
                    wp = lo.work_page_tokens
                    assert lo.ring_pages_per_warp >= 1, (kv, D, bs, hq, n)
                    row_bytes = D * {B.PA_F16: 2, B.PA_BF16: 2, B.PA_E4M3: 1, B.PA_INT8: 1, B.PA_INT4: 0.5}[kv]
                    R = (hq // 8) * n
                    if kv == B.PA_E4M3 and D == 256 and R % 16 == 0 and 16 <= R <= 64 and bs in (16, 32, 64, 128):
                        # the tensor-core kernel: 128-token chunks, every row of a kv head in one segment
                        assert wp == 128 and lo.rows_per_segment == R and lo.row_blocks == 1
                        assert lo.warps == lo.grid_ctas and lo.ring_pages_per_warp in (2, 3) and lo.group_size == 1
                        continue
                    if wp > bs:  # merged blocks
                        assert bs == 16 and wp == 32 and row_bytes <= 64 and lo.ring_pages_per_warp >= 2
                    else:
                        assert wp % 16 == 0 and bs % wp == 0, (kv, D, bs, hq, n)
                    if bs == 16 and row_bytes > 64:
                        assert wp == 16


# ------------------------------------------------------------- pa_insert


def _insert_status(B, p, src=None, ptrs=None, dev_error=None):
    """pa_insert's status for problem p with fake (never dereferenced) device
    pointers; every case here fails validation or has nothing to write, so
    nothing is launched."""
    a = 1 << 20                       # 16-byte aligned stand-ins
    d = dict(k_new=a, v_new=a, table=a, lens=a, ks=a, vs=a, kp=a, vp=a)
    d.update(ptrs or {})
    return B.raw_status("pa_insert", ctypes.byref(p), B.PA_BF16 if src is None else src, d["k_new"], d["v_new"],
                        d["table"], d["lens"], d["ks"], d["vs"], d["kp"], d["vp"], dev_error, None)


def test_insert_header_and_export(B):
    assert "pa_insert" in declared_symbols()
    assert hasattr(ctypes.CDLL(B.LIB_PATH), "pa_insert")


def test_insert_empty_batch_is_a_no_op(B):
    assert _insert_status(B, _prob(B, batch=0)) == B.PA_OK


@pytest.mark.parametrize("case,expect", [
    (dict(src=7), "INVALID_ARG"),                                     # unknown source dtype
    (dict(p=dict(next_n=0)), "INVALID_ARG"),
    (dict(p=dict(num_kv_heads=0)), "INVALID_ARG"),
    (dict(p=dict(kv_dtype=9)), "INVALID_ARG"),
    (dict(p=dict(k_scale_mode=5)), "INVALID_ARG"),
    (dict(p=dict(head_dim_k=100, head_dim_v=100)), "UNSUPPORTED"),        # not a multiple of 8
    (dict(p=dict(head_dim_k=4096, head_dim_v=4096)), "UNSUPPORTED"),      # beyond 2048 channels
    (dict(p=dict(k_scale_mode=3, v_scale_mode=3)), "UNSUPPORTED"),        # per-token scales: E4M3 only
    (dict(p=dict(kv_dtype=4, k_scale_mode=2, v_scale_mode=2), ptrs=dict(ks=None)), "INVALID_ARG"),
    (dict(p=dict(kv_dtype=4, k_scale_mode=2, v_scale_mode=2), ptrs=dict(vs=(1 << 20) + 4)), "INVALID_ARG"),
    (dict(p=dict(kv_dtype=3, k_scale_mode=1, v_scale_mode=1), ptrs=dict(ks=(1 << 20) + 2)), "INVALID_ARG"),
    (dict(ptrs=dict(k_new=(1 << 20) + 8)), "INVALID_ARG"),                # 16-byte alignment
    (dict(ptrs=dict(vp=(1 << 20) + 8)), "INVALID_ARG"),
    (dict(ptrs=dict(kp=None)), "INVALID_ARG"),
    (dict(ptrs=dict(table=None)), "INVALID_ARG"),
    (dict(ptrs=dict(lens=None)), "INVALID_ARG"),
    (dict(dev_error=(1 << 20) + 2), "INVALID_ARG"),
    (dict(p=dict(kv_dtype=3, k_scale_mode=3, v_scale_mode=3, block_size=3, num_kv_heads=1, head_dim_k=8,
                 head_dim_v=8)), "UNSUPPORTED"),                          # blocks not 16-byte multiples
    (dict(p=dict(v_is_k_prefix=1, head_dim_k=64, head_dim_v=128)), "INVALID_ARG"),
    (dict(p=dict(batch=1 << 20, next_n=1 << 10, num_kv_heads=8)), "UNSUPPORTED"),   # > 2^31 rows
])
def test_insert_rejects_bad_arguments(B, case, expect):
    p = _prob(B, **case.get("p", {}))
    st = _insert_status(B, p, case.get("src"), case.get("ptrs"), case.get("dev_error"))
    assert st == getattr(B, "PA_ERR_" + expect)


# --------------------------------------------------------- pa_sparse_attention


def _sparse_status(B, p, top_k=16, ws_bytes=1 << 20, ptrs=None):
    """pa_sparse_attention's status with fake (never dereferenced) device
    pointers; every case here fails validation or has no rows, so nothing is
    launched."""
    a = 1 << 20
    d = dict(sel=a, q=a, kp=a, vp=a, table=a, lens=a, ks=a, vs=a, ws=a, out=a, lse=a)
    d.update(ptrs or {})
    return B.raw_status("pa_sparse_attention", ctypes.byref(p), top_k, d["sel"], d["q"], d["kp"], d["vp"],
                        d["table"], d["lens"], d["ks"], d["vs"], d["ws"], ctypes.c_size_t(ws_bytes), d["out"],
                        d["lse"], None)


def test_sparse_header_and_workspace_size(B):
    assert {"pa_sparse_attention", "pa_sparse_workspace_size"} <= set(declared_symbols())
    p = _prob(B, batch=3, next_n=2)
    n = B.pa_sparse_workspace_size(p, 100)
    # error word, then per-token counts, then the token lists (256-byte aligned)
    assert n == 256 + 256 + ((3 * 2 * 100 * 4 + 255) // 256) * 256
    assert B.pa_sparse_workspace_size(_prob(B, batch=0), 100) == 256      # the error word only


def test_sparse_empty_batch_is_a_no_op(B):
    assert _sparse_status(B, _prob(B, batch=0)) == B.PA_OK


@pytest.mark.parametrize("case,expect", [
    (dict(top_k=-1), "INVALID_ARG"),
    (dict(p=dict(q_dtype=0)), "INVALID_ARG"),                                       # f32 queries
    (dict(p=dict(head_dim_k=96, head_dim_v=96)), "UNSUPPORTED"),
    (dict(p=dict(head_dim_v=64)), "UNSUPPORTED"),                                   # Dk != Dv
    (dict(p=dict(num_q_heads=136, num_kv_heads=8)), "UNSUPPORTED"),                  # 17 heads per kv head
    (dict(p=dict(head_dim_k=256, head_dim_v=256, num_q_heads=72, num_kv_heads=8)), "UNSUPPORTED"),  # 9 > 8
    (dict(p=dict(v_is_k_prefix=1)), "UNSUPPORTED"),
    (dict(p=dict(k_scale_mode=3, v_scale_mode=3)), "UNSUPPORTED"),                   # token scales: E4M3 only
    (dict(p=dict(max_context_len=1 << 21)), "UNSUPPORTED"),                         # planner bitmap > 227 KB
    (dict(ws_bytes=256), "WORKSPACE"),
    (dict(ptrs=dict(ws=(1 << 20) + 16)), "WORKSPACE"),
    (dict(ptrs=dict(sel=None)), "INVALID_ARG"),
    (dict(ptrs=dict(out=None)), "INVALID_ARG"),
    (dict(ptrs=dict(kp=(1 << 20) + 8)), "INVALID_ARG"),
    (dict(p=dict(kv_dtype=4, k_scale_mode=2, v_scale_mode=2), ptrs=dict(vs=None)), "INVALID_ARG"),
])
def test_sparse_rejects_bad_arguments(B, case, expect):
    p = _prob(B, **case.get("p", {}))
    st = _sparse_status(B, p, case.get("top_k", 16), case.get("ws_bytes", 1 << 20), case.get("ptrs"))
    assert st == getattr(B, "PA_ERR_" + expect)


# ------------------------------------------------- the header from plain C


def test_header_compiles_as_c11_and_links(B, tmp_path):
    import subprocess
    exe = tmp_path / "abi_check"
    src = os.path.join(ROOT, "tests", "c", "abi_check.c")
    libdir = os.path.dirname(B.LIB_PATH)
    r = subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I",
                        os.path.join(ROOT, "include"), src, "-o", str(exe), "-L", libdir, "-lpa",
                        "-Wl,-rpath," + libdir], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True)
    assert run.returncode == 0, run.stdout + run.stderr
    assert "version" in run.stdout


def _prototype_arity():
    """Argument count of every PA_API prototype in include/pa.h."""
    hdr = open(os.path.join(ROOT, "include", "pa.h")).read()
    hdr = re.sub(r"/\*.*?\*/", "", hdr, flags=re.S)
    out = {}
    for m in re.finditer(r"PA_API\s+[\w\s\*]+?\b(pa_\w+)\s*\(([^)]*)\)\s*;", hdr):
        args = m.group(2).strip()
        out[m.group(1)] = 0 if args in ("", "void") else len(args.split(","))
    return out


def test_binding_declares_every_prototype_with_its_arity(B):
    arity = _prototype_arity()
    assert len(arity) == len(declared_symbols())
    for name, n in arity.items():
        f = getattr(B._lib, name)
        assert f.argtypes is not None and len(f.argtypes) == n, (name, n, f.argtypes)


def _fp4(B, **kw):
    base = dict(batch=4, next_n=2, num_heads=64, head_dim=128, sf_vec_size=32, block_size=64, num_blocks=100,
                max_blocks_per_seq=16, max_context_len=1000, out_dtype=B.PA_BF16, out_stride=0, causal=1, rectify=0,
                sf_interleaved=0, num_sms=152, grid_ctas=0)
    base.update(kw)
    return B.Fp4Problem(**base)


def test_fp4_workspace_and_shapes(B):
    assert B.pa_fp4_logits_workspace_size(_fp4(B)) == 256 + 256 + 4 * 2 * 512
    for kw in (dict(head_dim=64), dict(sf_vec_size=16), dict(block_size=48), dict(num_heads=24),
               dict(next_n=4), dict(batch=1 << 20, max_blocks_per_seq=1 << 14)):
        st = B.raw_status("pa_fp4_logits_workspace_size", ctypes.byref(_fp4(B, **kw)), ctypes.byref(ctypes.c_size_t()))
        assert st == B.PA_ERR_UNSUPPORTED, kw
    for kw in (dict(batch=-1), dict(next_n=0), dict(out_dtype=B.PA_E4M3), dict(causal=2), dict(out_stride=999),
               dict(max_context_len=-1)):
        st = B.raw_status("pa_fp4_logits_workspace_size", ctypes.byref(_fp4(B, **kw)), ctypes.byref(ctypes.c_size_t()))
        assert st == B.PA_ERR_INVALID_ARG, kw


def test_fp4_rejects_bad_pointers_before_any_launch(B):
    p = _fp4(B)
    args = [0x10000, 0x20000, 0x30000, 0x40000, 0x50000, 0x60000]   # q, sf_q, kv, weights, lens, table
    n = B.pa_fp4_logits_workspace_size(p)
    assert B.raw_status("pa_fp4_logits", ctypes.byref(p), *args, None, n, 0x70000, None) == B.PA_ERR_WORKSPACE
    assert B.raw_status("pa_fp4_logits", ctypes.byref(p), *args, 0x80010, n, 0x70000, None) == B.PA_ERR_WORKSPACE
    assert B.raw_status("pa_fp4_logits", ctypes.byref(p), *args, 0x80000, n - 1, 0x70000, None) == B.PA_ERR_WORKSPACE
    bad_q = [0x10008] + args[1:]
    assert B.raw_status("pa_fp4_logits", ctypes.byref(p), *bad_q, 0x80000, n, 0x70000, None) == B.PA_ERR_INVALID_ARG
    no_kv = args[:2] + [None] + args[3:]
    assert B.raw_status("pa_fp4_logits", ctypes.byref(p), *no_kv, 0x80000, n, 0x70000, None) == B.PA_ERR_INVALID_ARG


def test_fp4_empty_batch_is_a_no_op(B):
    p = _fp4(B, batch=0)
    assert B.raw_status("pa_fp4_logits", ctypes.byref(p), None, None, None, None, None, None, 0x80000, 512,
                        None, None) == B.PA_OK
