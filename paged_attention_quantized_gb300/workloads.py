"""Seeded synthetic inputs for paged decode / verify attention.

This module only *draws* inputs: context lengths, physical block ids, queries,
quantized KV codes, scales, and the poisoning / relocation transforms.  It holds
none of the attention arithmetic and is shared, unchanged, by the CUDA path's
tests and benchmark and by the CPU oracle's tests.

Workload recipes (shapes and value distributions) follow the five benchmark
configurations of this library:

  tiny     fp16 decode, B=2, L={37,70}, Hq/Hkv=4/1, D=64, bs=16, 12 blocks
  bf16     bf16 GQA decode, B=64, L~U[512,8192], 32/8 heads, D=128, bs=16
  e4m3     E4M3 verify, B=32, L~U[1024,32768], next_n=4 causal, 32/8, D=256,
           bs=32, per-tensor scales 0.05, NaN-poisoned null/slack/padding
  int8     INT8 per-channel, B=128, L~U[2048,16384], 64/8, D=128, bs=16
  int4     the same with INT4 codes packed two per byte
  latent   single-latent MQA, B=256, L~lognormal(median 8192, sigma 1,
           cap 131072), next_n=2, 128/1 heads, Dk=576, Dv=512 (= first 512
           channels of K), bs=64, E4M3 with a per-token fp32 scale
  verify   the e4m3 recipe with next_n=16 (16 draft tokens verified per
           request: 64 query rows per kv head)
  qsa      sparse (selected-token) attention: four 64K-token requests, 256
           causal query rows each, 6 q / 1 kv heads, D=256, bs=16, fp16 KV
           (selections from make_selection)

Pool layout: every block is [Hkv][bs][row_bytes] codes; with per-token scales
the block continues with [Hkv][bs] fp32 scales.  INT4 stores channel 2i in the
low nibble of byte i.  Block 0 is the null block and is never referenced by a
real token.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional

import numpy as np
import torch

BITS = {"f16": 16, "bf16": 16, "e4m3": 8, "int8": 8, "int4": 4}
TORCH_FLOAT = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}

CONFIG_NAMES = ("tiny", "bf16", "e4m3", "int8", "int4", "latent")
# seed = 1234 + index of the configuration in the benchmark list (int8 and int4
# are the two halves of the fourth configuration and share its seed)
CONFIG_SEED = {"tiny": 1234, "bf16": 1235, "e4m3": 1236, "int8": 1237, "int4": 1237, "latent": 1238,
               "qsa": 1239, "verify": 1236}


@dataclass
class Workload:
    name: str
    B: int
    n: int
    Hq: int
    Hkv: int
    Dk: int
    Dv: int
    bs: int
    num_blocks: int
    max_blocks_per_seq: int
    max_context_len: int
    q_dtype: str
    kv_dtype: str
    out_dtype: str
    k_scale_mode: str
    v_scale_mode: str
    softmax_scale: float
    causal: bool
    v_is_k_prefix: bool
    q: torch.Tensor
    k_pool: torch.Tensor
    v_pool: Optional[torch.Tensor]
    block_table: torch.Tensor
    context_lens: torch.Tensor
    k_scale: Optional[torch.Tensor]
    v_scale: Optional[torch.Tensor]
    slack_ids: torch.Tensor = field(default=None)  # physical ids no token references
    seed: int = 0

    # -- derived sizes -----------------------------------------------------
    @property
    def k_row_bytes(self) -> int:
        return self.Dk * BITS[self.kv_dtype] // 8

    @property
    def v_row_bytes(self) -> int:
        return self.Dv * BITS[self.kv_dtype] // 8

    @property
    def rows_per_kv_head(self) -> int:
        return (self.Hq // self.Hkv) * self.n

    def effective_kv_bytes(self) -> int:
        """Algorithmic bytes one pass must read: real tokens only, codes plus
        scales, K and V once (a shared K/V plane counts once)."""
        L = int(self.context_lens.sum().item())
        per_tok = self.Hkv * self.k_row_bytes
        if self.k_scale_mode == "token":
            per_tok += self.Hkv * 4
        if not self.v_is_k_prefix:
            per_tok += self.Hkv * self.v_row_bytes
            if self.v_scale_mode == "token":
                per_tok += self.Hkv * 4
        return L * per_tok

    def to(self, device) -> "Workload":
        mv = lambda t: None if t is None else t.to(device)
        return replace(self, q=mv(self.q), k_pool=mv(self.k_pool), v_pool=mv(self.v_pool),
                       block_table=mv(self.block_table), context_lens=mv(self.context_lens),
                       k_scale=mv(self.k_scale), v_scale=mv(self.v_scale),
                       slack_ids=mv(self.slack_ids))


def block_bytes(Hkv: int, bs: int, row_bytes: int, token_scaled: bool) -> int:
    return Hkv * bs * row_bytes + (Hkv * bs * 4 if token_scaled else 0)


# ----------------------------------------------------------------- encoders


def e4m3_codes(x: torch.Tensor) -> torch.Tensor:
    """Round-to-nearest-even E4M3 codes of x, saturated to +-448 (never NaN)."""
    return x.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)


def pack_int4(codes: torch.Tensor) -> torch.Tensor:
    """Pack signed 4-bit codes [..., D] into bytes [..., D/2]; channel 2i goes
    to the low nibble of byte i (two's complement)."""
    u = (codes.to(torch.int16) & 0xF).to(torch.uint8)
    return (u[..., 0::2] | (u[..., 1::2] << 4)).contiguous()


# ----------------------------------------------------------------- helpers


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _poison_bytes(shape, gen, device) -> torch.Tensor:
    """Random bytes with a forced share of E4M3 NaN encodings (0x7F / 0xFF)."""
    b = torch.randint(0, 256, shape, generator=gen, device=device, dtype=torch.int16).to(torch.uint8)
    pick = torch.rand(shape, generator=gen, device=device) < 0.15
    nanv = torch.where(torch.rand(shape, generator=gen, device=device) < 0.5,
                       torch.tensor(0x7F, dtype=torch.uint8, device=device),
                       torch.tensor(0xFF, dtype=torch.uint8, device=device))
    return torch.where(pick, nanv, b)


def _lengths(name: str, B: int, gen_cpu: torch.Generator, lo=None, hi=None) -> torch.Tensor:
    if name == "tiny" and lo is None and hi is None and B <= 2:
        return torch.tensor([37, 70], dtype=torch.int32)[:B]
    if name == "qsa" and lo is None and hi is None:
        return torch.full((B,), 65536, dtype=torch.int32)
    if name == "latent":
        # lognormal, median 8192, sigma 1, capped at 131072, at least next_n
        z = torch.randn(B, generator=gen_cpu, dtype=torch.float64)
        L = torch.exp(math.log(8192.0) + 1.0 * z)
        lo_ = 2 if lo is None else lo
        hi_ = 131072 if hi is None else hi
        return L.round().clamp(lo_, hi_).to(torch.int32)
    rng = {"tiny": (1, 100), "qsa": (1, 65536), "verify": (1024, 32768), "bf16": (512, 8192), "e4m3": (1024, 32768), "int8": (2048, 16384), "int4": (2048, 16384)}[name]
    lo_ = rng[0] if lo is None else lo
    hi_ = rng[1] if hi is None else hi
    return torch.randint(lo_, hi_ + 1, (B,), generator=gen_cpu, dtype=torch.int64).to(torch.int32)


_SHAPES = {
    #        B   n  Hq Hkv  Dk   Dv  bs   q      kv     out    kmode      vmode     causal vprefix
    "tiny": (2, 1, 4, 1, 64, 64, 16, "f16", "f16", "f32", "none", "none", False, False),
    "bf16": (64, 1, 32, 8, 128, 128, 16, "bf16", "bf16", "bf16", "none", "none", False, False),
    "e4m3": (32, 4, 32, 8, 256, 256, 32, "bf16", "e4m3", "bf16", "tensor", "tensor", True, False),
    "int8": (128, 1, 64, 8, 128, 128, 16, "f16", "int8", "f32", "channel", "channel", False, False),
    "int4": (128, 1, 64, 8, 128, 128, 16, "f16", "int4", "f32", "channel", "channel", False, False),
    "latent": (256, 2, 128, 1, 576, 512, 64, "bf16", "e4m3", "bf16", "token", "token", True, True),
    # verify of 16 draft tokens per request (many query rows per kv head: 4 row blocks)
    "verify": (32, 16, 32, 8, 256, 256, 32, "bf16", "e4m3", "bf16", "tensor", "tensor", True, False),
    # sparse (selected-token) attention: four 64K-token requests, 256 query rows each
    "qsa": (4, 256, 6, 1, 256, 256, 16, "f16", "f16", "f16", "none", "none", True, False),
}


def make(name: str, device="cpu", seed: Optional[int] = None, *, B: Optional[int] = None,
         L_lo: Optional[int] = None, L_hi: Optional[int] = None, context_lens=None,
         poison: Optional[bool] = None, slack_frac: float = 0.10, n: Optional[int] = None,
         Hq: Optional[int] = None, Hkv: Optional[int] = None, D: Optional[int] = None,
         token_scale_spread: int = 0, bs: Optional[int] = None) -> Workload:
    """Draw one workload.  `name` picks the recipe; keyword overrides shrink it
    (batch, length range, explicit lengths, heads, head dim, block size) for
    tests.  Everything is a
    deterministic function of (name, seed, overrides, device).

    token_scale_spread = k > 0 (per-token E4M3 scales only): every block's
    scales are multiplied by 2^u, u uniform in {0..k} per block, and its codes
    encoded against them, so the scales of neighbouring pages differ by up
    to 2^k while the dequantized values keep their distribution."""
    if name not in _SHAPES:
        raise ValueError(f"unknown workload {name!r}")
    (B0, n0, Hq0, Hkv0, Dk, Dv, bs0, qd, kvd, outd, kmode, vmode, causal, vprefix) = _SHAPES[name]
    seed = CONFIG_SEED[name] if seed is None else seed
    B = B0 if B is None else B
    n = n0 if n is None else n
    Hq = Hq0 if Hq is None else Hq
    Hkv = Hkv0 if Hkv is None else Hkv
    if D is not None:
        if vprefix:
            raise ValueError("the latent recipe has fixed head dims")
        Dk = Dv = D
    if bs is not None:
        if vprefix:
            raise ValueError("the latent recipe has a fixed block size")
        bs = int(bs)
    else:
        bs = bs0
    poison = (name in ("e4m3", "verify")) if poison is None else poison
    device = torch.device(device)
    gcpu = _gen("cpu", seed)
    gdev = _gen(device, seed + 1)

    if context_lens is not None:
        L = torch.as_tensor(context_lens, dtype=torch.int32).cpu()
        B = int(L.numel())
    else:
        L = _lengths(name, B, gcpu, L_lo, L_hi)
    pages = [(int(l) + bs - 1) // bs for l in L.tolist()]
    W = sum(pages)
    if name == "tiny" and context_lens is None and B == 2:
        num_blocks = 12
    else:
        num_blocks = 1 + W + max(1, int(math.ceil(slack_frac * W)))
    mbps = max(1, max(pages) if pages else 1)
    max_ctx = max(1, int(L.max().item()) if B else 1)

    # physical ids: a seeded permutation of 1..num_blocks-1, assigned to the
    # logical pages in order; the remainder is slack
    perm = torch.randperm(num_blocks - 1, generator=gcpu).to(torch.int32) + 1
    table = torch.zeros((max(B, 1), mbps), dtype=torch.int32)
    ofs = 0
    for b in range(B):
        table[b, : pages[b]] = perm[ofs: ofs + pages[b]]
        ofs += pages[b]
    slack = perm[W:].clone()
    if poison:
        # unused table columns hold random valid ids: the null block or slack
        choices = torch.cat([torch.zeros(1, dtype=torch.int32), slack])
        for b in range(B):
            k = mbps - pages[b]
            if k > 0:
                idx = torch.randint(0, choices.numel(), (k,), generator=gcpu)
                table[b, pages[b]:] = choices[idx]
    table = table[:B] if B else table[:0]

    k_tok = kmode == "token"
    v_tok = vmode == "token"
    k_row = Dk * BITS[kvd] // 8
    v_row = Dv * BITS[kvd] // 8
    kbb = block_bytes(Hkv, bs, k_row, k_tok)
    vbb = block_bytes(Hkv, bs, v_row, v_tok)

    # queries
    qscale = 100.0 if name in ("int8", "int4") else 1.0
    q = (torch.randn((B, n, Hq, Dk), generator=gdev, device=device) * qscale).to(TORCH_FLOAT[qd])

    def fill_pool(row_bytes: int, D: int, tok: bool, is_k: bool, bb: int) -> torch.Tensor:
        pool = torch.zeros((num_blocks, bb), dtype=torch.uint8, device=device)
        codes_bytes = Hkv * bs * row_bytes
        ids = perm[:W].to(device=device, dtype=torch.int64)
        nb = ids.numel()
        if nb:
            # fill every referenced block fully in chunks (bounded temporaries)
            step = max(1, (1 << 26) // max(1, Hkv * bs * D))
            for s0 in range(0, nb, step):
                sel = ids[s0: s0 + step]
                m = sel.numel()
                shape = (m, Hkv, bs, D)
                if kvd in ("f16", "bf16"):
                    x = torch.randn(shape, generator=gdev, device=device).to(TORCH_FLOAT[kvd])
                    data = x.view(torch.uint8).reshape(m, codes_bytes)
                    sc = None
                elif kvd == "e4m3" and not tok:
                    x = torch.randn(shape, generator=gdev, device=device)
                    data = e4m3_codes(x / 0.05).reshape(m, codes_bytes)
                    sc = None
                elif kvd == "e4m3" and tok:
                    x = torch.randn(shape, generator=gdev, device=device)
                    s = x.abs().amax(dim=-1) / 448.0
                    s = torch.where(s > 0, s, torch.ones_like(s))
                    if token_scale_spread > 0:
                        u = torch.randint(0, token_scale_spread + 1, (m, 1, 1), generator=gdev, device=device)
                        s = s * torch.pow(2.0, u.to(s.dtype))
                    data = e4m3_codes(x / s[..., None]).reshape(m, codes_bytes)
                    sc = s.to(torch.float32).reshape(m, Hkv * bs)
                elif kvd in ("int8", "int4"):
                    lim = 127 if kvd == "int8" else 7
                    c = torch.randint(-lim, lim + 1, shape, generator=gdev, device=device, dtype=torch.int16)
                    if is_k:
                        zero = torch.rand((m, Hkv, bs, 1), generator=gdev, device=device) < 0.05
                        c = torch.where(zero, torch.zeros_like(c), c)
                    if kvd == "int8":
                        data = c.to(torch.int8).view(torch.uint8).reshape(m, codes_bytes)
                    else:
                        data = pack_int4(c).reshape(m, codes_bytes)
                    sc = None
                else:
                    raise ValueError(kvd)
                pool[sel, :codes_bytes] = data
                if tok:
                    pool[sel, codes_bytes:] = sc.contiguous().view(torch.uint8).reshape(m, -1)
        if poison:
            unref = torch.cat([torch.zeros(1, dtype=torch.int64), slack.to(torch.int64)]).to(device)
            nun = unref.numel()
            hybrid = torch.rand(nun, generator=gdev, device=device) < 0.20
            hybrid[0] = False
            junk = _poison_bytes((nun, bb), gdev, device)
            state = torch.randn((nun, bb // 2), generator=gdev, device=device).to(torch.float16)
            state = state.view(torch.uint8).reshape(nun, -1)
            if state.shape[1] < bb:
                state = torch.cat([state, junk[:, state.shape[1]:]], dim=1)
            pool[unref] = torch.where(hybrid[:, None], state, junk)
            # tail slots of each request's last, partial page
            for b in range(B):
                Lb = int(L[b])
                if Lb % bs == 0 or pages[b] == 0:
                    continue
                blk = int(table[b, pages[b] - 1])
                first = Lb % bs
                for g in range(Hkv):
                    lo = (g * bs + first) * row_bytes
                    hi = (g * bs + bs) * row_bytes
                    pool[blk, lo:hi] = _poison_bytes((hi - lo,), gdev, device)
                    if tok:
                        slo = codes_bytes + (g * bs + first) * 4
                        shi = codes_bytes + (g * bs + bs) * 4
                        pool[blk, slo:shi] = 0xFF
        return pool

    k_pool = fill_pool(k_row, Dk, k_tok, True, kbb)
    v_pool = None if vprefix else fill_pool(v_row, Dv, v_tok, False, vbb)

    k_scale = v_scale = None
    if kmode == "tensor":
        k_scale = torch.tensor([0.05], dtype=torch.float32, device=device)
    if vmode == "tensor" and not vprefix:
        v_scale = torch.tensor([0.05], dtype=torch.float32, device=device)
    if kmode == "channel":
        k_scale = torch.pow(10.0, torch.rand((Hkv, Dk), generator=gdev, device=device) * 5.0 - 2.0).float()
    if vmode == "channel" and not vprefix:
        v_scale = torch.pow(10.0, torch.rand((Hkv, Dv), generator=gdev, device=device) * 5.0 - 2.0).float()

    return Workload(
        name=name, B=B, n=n, Hq=Hq, Hkv=Hkv, Dk=Dk, Dv=Dv, bs=bs, num_blocks=num_blocks,
        max_blocks_per_seq=mbps, max_context_len=max_ctx, q_dtype=qd, kv_dtype=kvd, out_dtype=outd,
        k_scale_mode=kmode, v_scale_mode=vmode if not vprefix else kmode,
        softmax_scale=1.0 / math.sqrt(Dk), causal=causal, v_is_k_prefix=vprefix,
        q=q, k_pool=k_pool, v_pool=v_pool, block_table=table.to(device), context_lens=L.to(device),
        k_scale=k_scale, v_scale=v_scale, slack_ids=slack.to(device), seed=seed)


# ---------------------------------------------------------------- transforms


def relocate(w: Workload, seed: int) -> Workload:
    """Move every non-null block to a new physical id (a seeded permutation of
    1..num_blocks-1, block 0 stays the null block) and rewrite the table to
    match.  Logical contents are unchanged."""
    g = _gen("cpu", seed)
    pi = torch.cat([torch.zeros(1, dtype=torch.int64),
                    torch.randperm(w.num_blocks - 1, generator=g).to(torch.int64) + 1])
    dev = w.k_pool.device
    pi_d = pi.to(dev)
    inv = torch.empty_like(pi_d)
    inv[pi_d] = torch.arange(w.num_blocks, device=dev)

    def move(pool):
        return None if pool is None else pool.index_select(0, inv).contiguous()

    table = pi_d.index_select(0, w.block_table.reshape(-1).to(torch.int64)).to(torch.int32)
    table = table.reshape(w.block_table.shape)
    slack = pi_d.index_select(0, w.slack_ids.to(torch.int64)).to(torch.int32)
    return replace(w, k_pool=move(w.k_pool), v_pool=move(w.v_pool), block_table=table, slack_ids=slack)


def poison_unreferenced(w: Workload, seed: int) -> Workload:
    """Overwrite every byte that no visible token maps to (null block, slack
    blocks, tail slots of last pages) with random bytes that include E4M3 NaN
    encodings, and point unused table columns at the null block or slack."""
    g = _gen("cpu", seed)
    gdev = _gen(w.k_pool.device, seed + 7)
    dev = w.k_pool.device
    L = w.context_lens.cpu().tolist()
    pages = [(l + w.bs - 1) // w.bs for l in L]
    k_tok = w.k_scale_mode == "token"
    v_tok = (w.v_scale_mode == "token")

    def pz(pool, row_bytes, tok):
        if pool is None:
            return None
        pool = pool.clone()
        codes = w.Hkv * w.bs * row_bytes
        unref = torch.cat([torch.zeros(1, dtype=torch.int64, device=dev), w.slack_ids.to(torch.int64)])
        pool[unref] = _poison_bytes((unref.numel(), pool.shape[1]), gdev, dev)
        tab = w.block_table.cpu()
        for b, Lb in enumerate(L):
            if Lb % w.bs == 0 or pages[b] == 0:
                continue
            blk = int(tab[b, pages[b] - 1])
            first = Lb % w.bs
            for h in range(w.Hkv):
                lo, hi = (h * w.bs + first) * row_bytes, (h * w.bs + w.bs) * row_bytes
                pool[blk, lo:hi] = _poison_bytes((hi - lo,), gdev, dev)
                if tok:
                    pool[blk, codes + (h * w.bs + first) * 4: codes + (h * w.bs + w.bs) * 4] = 0xFF
        return pool

    table = w.block_table.cpu().clone()
    choices = torch.cat([torch.zeros(1, dtype=torch.int32), w.slack_ids.cpu().to(torch.int32)])
    for b in range(w.B):
        k = w.max_blocks_per_seq - pages[b]
        if k > 0:
            idx = torch.randint(0, choices.numel(), (k,), generator=g)
            table[b, pages[b]:] = choices[idx]
    return replace(w, k_pool=pz(w.k_pool, w.k_row_bytes, k_tok),
                   v_pool=pz(w.v_pool, w.v_row_bytes, v_tok), block_table=table.to(dev))


def referenced_mask(w: Workload) -> np.ndarray:
    """[num_blocks] bool: blocks that hold at least one visible token."""
    m = np.zeros(w.num_blocks, dtype=bool)
    tab = w.block_table.cpu().numpy()
    for b, Lb in enumerate(w.context_lens.cpu().tolist()):
        p = (Lb + w.bs - 1) // w.bs
        m[tab[b, :p]] = True
    return m


# ------------------------------------------------------------ new KV rows


def new_kv_rows(w: Workload, src: str = "bf16", seed: int = 0, device=None, outliers: bool = True):
    """Seeded new K / V rows [B, n, Hkv, D] for an insert into w's pool, in the
    source dtype `src` ("f32", "f16" or "bf16"); V is None when it is the
    prefix of the K plane.

    Value recipe, per cache encoding: 16-bit caches N(0,1); per-tensor E4M3
    N(0,1) with 1% of the values times 100 (past the +-448 code range at the
    0.05 scale); per-channel INT8 / INT4 N(0, (c * k_scale[g, d])^2) with
    c = 127/3 or 7/3, 1% of the values times 10 (clamped codes); per-token
    E4M3 N(0,1) times 10^U(-3,3) per row, 2% of the rows all zero.  With
    outliers=False the values follow the pool's own recipe instead (N(0,1),
    or N(0, (c * k_scale[g, d])^2) for per-channel integer caches)."""
    device = w.k_pool.device if device is None else torch.device(device)
    g = _gen(device, seed)
    dt = TORCH_FLOAT[src]

    def rows(D, scale, mode):
        shape = (w.B, w.n, w.Hkv, D)
        x = torch.randn(shape, generator=g, device=device)
        if not outliers:
            if w.kv_dtype in ("int8", "int4") and mode == "channel":
                c = (127.0 if w.kv_dtype == "int8" else 7.0) / 3.0
                x = x * c * scale.to(device).float().reshape(1, 1, w.Hkv, D)
        elif w.kv_dtype == "e4m3" and mode == "tensor":
            big = torch.rand(shape, generator=g, device=device) < 0.01
            x = torch.where(big, x * 100.0, x)
        elif w.kv_dtype in ("int8", "int4") and mode == "channel":
            c = (127.0 if w.kv_dtype == "int8" else 7.0) / 3.0
            x = x * c * scale.to(device).float().reshape(1, 1, w.Hkv, D)
            big = torch.rand(shape, generator=g, device=device) < 0.01
            x = torch.where(big, x * 10.0, x)
        elif mode == "token":
            mag = torch.pow(10.0, torch.rand((w.B, w.n, w.Hkv, 1), generator=g, device=device) * 6.0 - 3.0)
            zero = torch.rand((w.B, w.n, w.Hkv, 1), generator=g, device=device) < 0.02
            x = torch.where(zero, torch.zeros_like(x), x * mag)
        return x.to(dt).contiguous()

    k = rows(w.Dk, w.k_scale, w.k_scale_mode)
    v = None if w.v_is_k_prefix else rows(w.Dv, w.v_scale, w.v_scale_mode)
    return k, v


# ------------------------------------------------------- sparse selections


def make_selection(w: Workload, k: int, seed: int = 0, shared: float = 0.9, device=None) -> torch.Tensor:
    """Seeded token selections [B, next_n, k] int32 for sparse attention: the
    logical positions each query token attends to, in no particular order,
    -1 for unused entries.

    Recipe ("highly shared selections"): every request draws one pool of k
    positions uniformly from its tokens; each query row keeps a `shared`
    share of that pool and draws the rest from its own visible tokens (which
    may repeat pool entries), then the row is shuffled.  Rows whose visible
    length is below k list every visible token once and pad with -1."""
    device = w.context_lens.device if device is None else torch.device(device)
    g = _gen("cpu", seed)
    L = w.context_lens.cpu().tolist()
    out = torch.full((w.B, w.n, k), -1, dtype=torch.int32)
    for b, Lb in enumerate(L):
        pool = torch.randperm(max(Lb, 1), generator=g)[:k].to(torch.int32) if Lb > 0 else torch.zeros(0, dtype=torch.int32)
        for j in range(w.n):
            vis = Lb - (w.n - 1 - j) if w.causal else Lb
            if vis <= 0:
                continue
            if vis <= k:
                row = torch.randperm(vis, generator=g).to(torch.int32)
                out[b, j, :vis] = row
                continue
            keep = pool[pool < vis]
            nkeep = min(int(round(shared * k)), keep.numel())
            keep = keep[torch.randperm(keep.numel(), generator=g)[:nkeep]]
            rest = torch.randint(0, vis, (k - nkeep,), generator=g, dtype=torch.int64).to(torch.int32)
            row = torch.cat([keep, rest])
            out[b, j] = row[torch.randperm(k, generator=g)]
    return out.to(device)


# ------------------------------------------------ FP4 paged MQA logits


@dataclass
class Fp4Logits:
    """Inputs of FP4 (MXFP4) paged MQA logits (see make_fp4)."""
    name: str
    B: int
    n: int
    H: int
    D: int
    bs: int
    sf_vec: int
    num_blocks: int
    max_blocks_per_seq: int
    max_context_len: int
    out_dtype: str
    causal: bool
    rectify: bool
    sf_interleaved: bool
    q: torch.Tensor            # [B, n, H, D/2] uint8, two E2M1 values per byte
    sf_q: torch.Tensor         # [B, n, H] int32, D/sf_vec UE8M0 bytes
    kv_fused: torch.Tensor     # [num_blocks, bs * (D/2 + D/sf_vec)] uint8
    weights: torch.Tensor      # [B * n, H] float32
    block_table: torch.Tensor  # [B, max_blocks_per_seq] int32
    context_lens: torch.Tensor  # [B] int32
    seed: int = 0

    @property
    def row_bytes(self) -> int:
        return self.D // 2 + self.D // self.sf_vec

    def kv_bytes(self) -> int:
        """Algorithmic bytes read: every visible token's packed values and
        scale bytes once (the tokens of the longest row of each request)."""
        return int(self.context_lens.sum().item()) * self.row_bytes

    def out_bytes(self) -> int:
        es = {"f32": 4, "f16": 2, "bf16": 2}[self.out_dtype]
        return self.B * self.n * self.max_context_len * es

    def to(self, device) -> "Fp4Logits":
        mv = lambda t: None if t is None else t.to(device)
        return replace(self, q=mv(self.q), sf_q=mv(self.sf_q), kv_fused=mv(self.kv_fused),
                       weights=mv(self.weights), block_table=mv(self.block_table),
                       context_lens=mv(self.context_lens))


def _sf_words(shape, gen, device, lo: int, hi: int) -> torch.Tensor:
    """int32 words of four UE8M0 bytes, each uniform in [lo, hi]."""
    b = torch.randint(lo, hi + 1, shape + (4,), generator=gen, device=device, dtype=torch.int64)
    w = b[..., 0] | (b[..., 1] << 8) | (b[..., 2] << 16) | (b[..., 3] << 24)
    return torch.where(w >= 2 ** 31, w - 2 ** 32, w).to(torch.int32)


def make_fp4(device="cpu", seed: int = 1240, *, B: int = 128, n: int = 2, H: int = 64, D: int = 128,
             bs: int = 64, L_lo: int = 4096, L_hi: int = 65536, context_lens=None, causal: bool = True,
             rectify: bool = False, sf_interleaved: bool = False, out_dtype: str = "bf16",
             scale_lo: int = 124, scale_hi: int = 130, slack_frac: float = 0.10) -> Fp4Logits:
    """Seeded inputs for FP4 paged MQA logits.

    Recipe (the indexer shape of the FlashInfer fp4_paged_mqa_logits page:
    64 heads of dim 128, MXFP4 with 32-value UE8M0 groups, 64-token blocks):
    B requests, L ~ U[L_lo, L_hi], next_n query rows (causal: row j sees
    tokens up to L - n + j), every E2M1 code equally likely in q and K (all
    16, including -0), scale bytes uniform in [scale_lo, scale_hi], weights
    N(0, 1).  Physical ids a seeded permutation of 1..num_blocks-1; the table
    is as wide as the page's precondition round_up(L, 128) / bs asks, extra
    columns pointing at the null block or slack blocks; unreferenced blocks
    and the unused slots of last blocks hold random bytes (scale byte 0xFF,
    NaN, included)."""
    device = torch.device(device)
    gcpu = _gen("cpu", seed)
    gdev = _gen(device, seed + 1)
    if context_lens is not None:
        L = torch.as_tensor(context_lens, dtype=torch.int32).cpu()
        B = int(L.numel())
    else:
        L = torch.randint(L_lo, L_hi + 1, (B,), generator=gcpu, dtype=torch.int64).to(torch.int32)
    sf_vec = 32
    row = D // 2 + D // sf_vec
    pages = [(int(l) + bs - 1) // bs for l in L.tolist()]
    cols = [((int(l) + 127) // 128) * 128 // bs for l in L.tolist()]
    Wp = sum(pages)
    num_blocks = 1 + Wp + max(1, int(math.ceil(slack_frac * Wp)))
    mbps = max(1, max(cols) if cols else 1)
    max_ctx = max(1, int(L.max().item()) if B else 1)
    perm = torch.randperm(num_blocks - 1, generator=gcpu).to(torch.int32) + 1
    table = torch.zeros((max(B, 1), mbps), dtype=torch.int32)
    slack = perm[Wp:].clone()
    choices = torch.cat([torch.zeros(1, dtype=torch.int32), slack])
    ofs = 0
    for b in range(B):
        table[b, : pages[b]] = perm[ofs: ofs + pages[b]]
        ofs += pages[b]
        k = mbps - pages[b]
        if k > 0:
            table[b, pages[b]:] = choices[torch.randint(0, choices.numel(), (k,), generator=gcpu)]
    table = table[:B]

    q = torch.randint(0, 256, (B, n, H, D // 2), generator=gdev, device=device, dtype=torch.int16).to(torch.uint8)
    sf_q = _sf_words((B, n, H), gdev, device, scale_lo, scale_hi)
    weights = torch.randn((B * n, H), generator=gdev, device=device, dtype=torch.float32)

    # every block starts as junk (random bytes, scale bytes included); the
    # referenced slots are then written with codes and in-range scales
    kv = torch.randint(0, 256, (num_blocks, bs * row), generator=gdev, device=device,
                       dtype=torch.int16).to(torch.uint8)
    data = bs * (D // 2)
    nsf = D // sf_vec
    if sf_interleaved and bs % SF_WORD != 0:
        raise ValueError("interleaved scales need a block size divisible by 4")
    # word slot of each token inside the scale region
    slot_of = list(range(bs))
    if sf_interleaved:
        for k in range(bs):
            slot_of[(k % SF_WORD) * (bs // SF_WORD) + k // SF_WORD] = k
    slot_idx = torch.tensor(slot_of, dtype=torch.int64, device=device)
    ofs = 0
    for b in range(B):
        for p in range(pages[b]):
            blk = int(perm[ofs + p])
            ntok = min(bs, int(L[b]) - p * bs)
            kv[blk, : ntok * (D // 2)] = torch.randint(0, 256, (ntok * (D // 2),), generator=gdev, device=device,
                                                       dtype=torch.int16).to(torch.uint8)
            sc = torch.randint(scale_lo, scale_hi + 1, (ntok, nsf), generator=gdev, device=device,
                               dtype=torch.int16).to(torch.uint8)
            pos = data + slot_idx[:ntok, None] * nsf + torch.arange(nsf, device=device)[None, :]
            kv[blk].index_put_((pos.reshape(-1),), sc.reshape(-1))
        ofs += pages[b]
    return Fp4Logits(name="fp4", B=B, n=n, H=H, D=D, bs=bs, sf_vec=sf_vec, num_blocks=num_blocks,
                     max_blocks_per_seq=mbps, max_context_len=max_ctx, out_dtype=out_dtype, causal=causal,
                     rectify=rectify, sf_interleaved=sf_interleaved, q=q, sf_q=sf_q, kv_fused=kv,
                     weights=weights, block_table=table.to(device), context_lens=L.to(device), seed=seed)


SF_WORD = 4  # UE8M0 bytes in one scale word (one token's scales at D = 128)


def relocate_fp4(w: Fp4Logits, seed: int) -> Fp4Logits:
    """Move every non-null block of an Fp4Logits pool to a new physical id."""
    g = _gen("cpu", seed)
    pi = torch.cat([torch.zeros(1, dtype=torch.int64),
                    torch.randperm(w.num_blocks - 1, generator=g).to(torch.int64) + 1]).to(w.kv_fused.device)
    inv = torch.empty_like(pi)
    inv[pi] = torch.arange(w.num_blocks, device=pi.device)
    table = pi.index_select(0, w.block_table.reshape(-1).to(torch.int64)).to(torch.int32).reshape(w.block_table.shape)
    return replace(w, kv_fused=w.kv_fused.index_select(0, inv).contiguous(), block_table=table)
