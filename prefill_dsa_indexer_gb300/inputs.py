"""Seeded synthetic inputs for the DSA layer (shared by tests, smoke and bench).

This module holds no part of the layer's arithmetic (no scoring, selection or
attention).  It draws values with torch's seeded generators and stores them
in the cache byte formats the layer reads:

* index keys: 128 values per token, N(0,1), stored as FP8 e4m3 with one fp32
  scale per token (amax/448, 132 B/token), or as MXFP4 (e2m1 elements with
  one e8m0 scale per 32 values, 68 B/token);
* latents: 576 values per token (512 latent + 64 RoPE dims), N(0,1), stored
  as FP8 e4m3 with one per-tensor scale (amax/448 over the used pool,
  576 B/token), or as NVFP4 (512 e2m1 values with one e4m3 scale per 16
  values, plus the 64 RoPE dims in FP8 with the per-tensor scale,
  352 B/token);
* indexer query: 32 heads x 128 FP8 e4m3 values from N(0,1), no scale;
  head weights U(0,1) fp32;
* MLA query: 96 heads x 576 bf16 values from N(0,1).

Widths and encodings follow the vLLM blog "Day-0 support for Kimi K3.1 Pro"
(sections "Sparse attention in K3.1 Pro", "KV cache footprint", "One KV
cache, three states") and the OCP MX v1.0 rules for the shared scale
(exponent = floor(log2(amax)) - emax(e2m1), emax = 2).  Encoding uses torch's
float8_e4m3fn cast (round-to-nearest-even) and a round-to-nearest-even e2m1
table lookup.

Paging: every request's tokens live in 64-token pages drawn from a random
permutation of a pool that is larger than needed (free pages between
requests); slots that hold no token are filled with NaN codes so that a read
outside the valid data shows up as NaN.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

PAGE = 64
IDX_DIM, IDX_HEADS = 128, 32
LAT_DIM, V_DIM, ROPE_DIM = 576, 512, 64
KEY_FP8, KEY_MXFP4, LATENT_FP8, LATENT_NVFP4 = 1, 2, 3, 4

INDEX_TOKEN_BYTES = {KEY_FP8: IDX_DIM + 4, KEY_MXFP4: IDX_DIM // 2 + IDX_DIM // 32}
LATENT_TOKEN_BYTES = {LATENT_FP8: LAT_DIM, LATENT_NVFP4: V_DIM // 2 + V_DIM // 16 + ROPE_DIM}


def index_page_bytes(fmt: int) -> int:
    return PAGE * INDEX_TOKEN_BYTES[fmt]


def latent_page_bytes(fmt: int) -> int:
    return PAGE * LATENT_TOKEN_BYTES[fmt]


@dataclass
class Workload:
    """One DSA layer invocation: requests, their query rows and formats."""

    name: str
    ctx: list[int]               # cached tokens per request (incl. the query rows' own tokens)
    rows_per_req: int            # query rows per request (1 decode, 4 verify, n prefill)
    rows_per_group: int          # consecutive rows the indexer scores together
    key_fmt: int = KEY_FP8
    lat_fmt: int = LATENT_FP8
    k: int = 2048
    heads: int = 96
    seed: int = 0
    extra_pages: float = 0.25    # free pool pages, as a fraction of the used ones

    @property
    def num_rows(self) -> int:
        return len(self.ctx) * self.rows_per_req

    def row_ctx(self) -> np.ndarray:
        """Row i of request b sees L_b - n + 1 + i tokens (causal query rows)."""
        n = self.rows_per_req
        out = [L - n + 1 + i for L in self.ctx for i in range(n)]
        return np.asarray(out, dtype=np.int32)

    def row_req(self) -> np.ndarray:
        return np.repeat(np.arange(len(self.ctx), dtype=np.int32), self.rows_per_req)


def _ctx_uniform(seed: int, n: int, lo: int, hi: int) -> list[int]:
    rng = np.random.default_rng(seed)
    return [int(x) for x in rng.integers(lo, hi + 1, size=n)]


def workload(name: str) -> Workload:
    """The named workloads (sizes in tokens)."""
    if name == "decode_tiny_4k":
        return Workload(name, [4096], 1, 1, seed=1000, extra_pages=1.0)
    if name == "decode_b32_16k_64k":
        return Workload(name, _ctx_uniform(1001, 32, 16384, 65536), 1, 1, seed=1001)
    if name == "verify_b4_256k":
        return Workload(name, [262144] * 4, 4, 4, seed=1002)
    if name == "verify_b1_1m":
        return Workload(name, [1048576], 4, 4, seed=2002)
    if name == "decode_b8_128k_fp4":
        return Workload(name, [131072] * 8, 1, 1, KEY_MXFP4, LATENT_NVFP4, seed=1003)
    if name == "decode_b8_128k_fp8":
        return Workload(name, [131072] * 8, 1, 1, seed=1003)
    if name == "prefill_8k_on_56k":
        return Workload(name, [65536], 8192, 8, seed=1004)
    if name == "prefill_1k_on_15k":  # the prefill shape at an eighth of the rows (profiling size)
        return Workload(name, [16384], 1024, 8, seed=1005)
    raise KeyError(name)


WORKLOADS = ("decode_tiny_4k", "decode_b32_16k_64k", "verify_b4_256k", "verify_b1_1m",
             "decode_b8_128k_fp4", "decode_b8_128k_fp8", "prefill_8k_on_56k", "prefill_1k_on_15k")


@dataclass
class Inputs:
    wl: Workload
    idx_pool: torch.Tensor        # uint8 [num_pages, index_page_bytes]
    lat_pool: torch.Tensor        # uint8 [num_pages, latent_page_bytes]
    tensor_scale: float           # FP8 latent / RoPE per-tensor scale
    block_table: torch.Tensor     # int32 [B, max_pages]
    row_req: torch.Tensor         # int32 [R]
    row_ctx: torch.Tensor         # int32 [R]
    q_idx: torch.Tensor           # uint8 [R, 32, 128] e4m3 codes
    head_w: torch.Tensor          # float32 [R, 32]
    q_mla: torch.Tensor           # int16 [R, H, 576] bf16 bits
    extra: dict = field(default_factory=dict)

    @property
    def num_pages(self) -> int:
        return self.idx_pool.shape[0]

    @property
    def max_ctx(self) -> int:
        return max(self.wl.ctx)

    def np(self, name: str) -> np.ndarray:
        t = getattr(self, name)
        if name == "q_mla":
            return t.cpu().numpy().view(np.uint16)
        return t.cpu().numpy()

    def to(self, device) -> "Inputs":
        mv = {n: getattr(self, n).to(device) for n in
              ("idx_pool", "lat_pool", "block_table", "row_req", "row_ctx", "q_idx", "head_w", "q_mla")}
        return Inputs(self.wl, tensor_scale=self.tensor_scale, extra=dict(self.extra), **mv)


# ------------------------------------------------------------------ encoders

def e4m3_codes(x: torch.Tensor) -> torch.Tensor:
    """float -> e4m3 byte codes, round-to-nearest-even, saturated to +-448."""
    return x.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)


_E2M1_BOUNDS = (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)


def e2m1_codes(x: torch.Tensor) -> torch.Tensor:
    """float -> 4-bit e2m1 codes (uint8 holding one nibble), RNE, saturating.

    Magnitudes of codes 0..7 are 0, .5, 1, 1.5, 2, 3, 4, 6; a value halfway
    between two goes to the code with an even mantissa bit."""
    a = x.abs()
    b = torch.tensor(_E2M1_BOUNDS, dtype=a.dtype, device=a.device)
    code = torch.bucketize(a, b, right=False)
    tie_up = (a == 0.75) | (a == 1.75) | (a == 3.5)
    code = (code + tie_up.to(code.dtype)).clamp(max=7).to(torch.uint8)
    sign = (x < 0).to(torch.uint8) << 3
    return code | sign


def pack_nibbles(codes: torch.Tensor) -> torch.Tensor:
    """[..., 2n] nibbles -> [..., n] bytes, element 2j in the low nibble."""
    lo = codes[..., 0::2]
    hi = codes[..., 1::2]
    return lo | (hi << 4)


def mxfp4_encode(x: torch.Tensor):
    """x [T, 128] -> (packed [T, 64] uint8, e8m0 scales [T, 4] uint8)."""
    T = x.shape[0]
    blk = x.view(T, IDX_DIM // 32, 32)
    amax = blk.abs().amax(dim=-1)
    e = torch.floor(torch.log2(amax.clamp(min=1e-38))) - 2 + 127
    e = torch.where(amax > 0, e, torch.zeros_like(e)).clamp(0, 254)
    scale = torch.pow(2.0, e - 127)
    codes = e2m1_codes(blk / scale.unsqueeze(-1)).view(T, IDX_DIM)
    return pack_nibbles(codes), e.to(torch.uint8)


def nvfp4_encode(x: torch.Tensor):
    """x [T, 512] -> (packed [T, 256] uint8, e4m3 scales [T, 32] uint8)."""
    T = x.shape[0]
    blk = x.view(T, V_DIM // 16, 16)
    amax = blk.abs().amax(dim=-1)
    sc_codes = e4m3_codes(amax / 6.0)
    sc = sc_codes.view(torch.float8_e4m3fn).to(torch.float32)
    safe = torch.where(sc > 0, sc, torch.ones_like(sc))
    codes = e2m1_codes(blk / safe.unsqueeze(-1))
    codes = torch.where((sc > 0).unsqueeze(-1), codes, torch.zeros_like(codes)).view(T, V_DIM)
    return pack_nibbles(codes), sc_codes


# ------------------------------------------------------------------ builders

def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _paging(wl, page: int = PAGE):
    rng = np.random.default_rng(wl.seed * 7 + 1)
    npages = [(L + page - 1) // page for L in wl.ctx]
    used = sum(npages)
    total = used + max(1, int(used * wl.extra_pages))
    perm = rng.permutation(total).astype(np.int32)
    width = max(npages)
    bt = np.zeros((len(wl.ctx), width), dtype=np.int32)
    off = 0
    for b, n in enumerate(npages):
        bt[b, :n] = perm[off:off + n]
        off += n
    return bt, total


def token_slots(block_table: np.ndarray, ctx: list[int]) -> np.ndarray:
    """Physical slot of every cached token, requests concatenated."""
    out = []
    for b, L in enumerate(ctx):
        t = np.arange(L, dtype=np.int64)
        out.append(block_table[b, t // PAGE].astype(np.int64) * PAGE + t % PAGE)
    return np.concatenate(out)


def make_inputs(wl: Workload, device="cpu", chunk_tokens: int = 1 << 18) -> Inputs:
    device = torch.device(device)
    bt_np, num_pages = _paging(wl)
    slots = torch.from_numpy(token_slots(bt_np, wl.ctx)).to(device)
    T = slots.numel()
    pg = slots // PAGE
    j = slots % PAGE

    # ---- index pool
    ipb = index_page_bytes(wl.key_fmt)
    idx_pool = torch.full((num_pages, ipb), 0x7F, dtype=torch.uint8, device=device)
    gk = _gen(device, wl.seed * 100 + 1)
    if wl.key_fmt == KEY_FP8:
        codes_v = idx_pool[:, :PAGE * IDX_DIM].view(num_pages, PAGE, IDX_DIM)
        scale_v = idx_pool[:, PAGE * IDX_DIM:].view(torch.float32).view(num_pages, PAGE)
        scale_v.fill_(float("nan"))
    else:
        half = IDX_DIM // 2
        codes_v = idx_pool[:, :PAGE * half].view(num_pages, PAGE, half)
        scale_v = idx_pool[:, PAGE * half:].view(num_pages, PAGE, IDX_DIM // 32)
        scale_v.fill_(0xFF)
    for s0 in range(0, T, chunk_tokens):
        s1 = min(T, s0 + chunk_tokens)
        x = torch.randn((s1 - s0, IDX_DIM), generator=gk, device=device, dtype=torch.float32)
        p, jj = pg[s0:s1], j[s0:s1]
        if wl.key_fmt == KEY_FP8:
            amax = x.abs().amax(dim=-1)
            sc = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
            codes_v[p, jj] = e4m3_codes(x / sc.unsqueeze(-1))
            scale_v[p, jj] = sc
        else:
            packed, e = mxfp4_encode(x)
            codes_v[p, jj] = packed
            scale_v[p, jj] = e

    # ---- latent pool
    lpb = latent_page_bytes(wl.lat_fmt)
    lat_pool = torch.full((num_pages, lpb), 0x7F, dtype=torch.uint8, device=device)
    gl = _gen(device, wl.seed * 100 + 2)
    # per-tensor scale of the FP8 part: amax over all used latents / 448.
    # Pass 1 draws and records amax; pass 2 redraws the same stream.
    amax = torch.zeros((), device=device)
    for s0 in range(0, T, chunk_tokens):
        s1 = min(T, s0 + chunk_tokens)
        x = torch.randn((s1 - s0, LAT_DIM), generator=gl, device=device, dtype=torch.float32)
        part = x if wl.lat_fmt == LATENT_FP8 else x[:, V_DIM:]
        amax = torch.maximum(amax, part.abs().amax())
    tensor_scale = float(amax.item()) / 448.0 if float(amax.item()) > 0 else 1.0
    gl = _gen(device, wl.seed * 100 + 2)
    if wl.lat_fmt == LATENT_FP8:
        lat_v = lat_pool.view(num_pages, PAGE, LAT_DIM)
    else:
        hb = V_DIM // 2
        codes_l = lat_pool[:, :PAGE * hb].view(num_pages, PAGE, hb)
        sc_l = lat_pool[:, PAGE * hb:PAGE * (hb + V_DIM // 16)].view(num_pages, PAGE, V_DIM // 16)
        rope_l = lat_pool[:, PAGE * (hb + V_DIM // 16):].view(num_pages, PAGE, ROPE_DIM)
    for s0 in range(0, T, chunk_tokens):
        s1 = min(T, s0 + chunk_tokens)
        x = torch.randn((s1 - s0, LAT_DIM), generator=gl, device=device, dtype=torch.float32)
        p, jj = pg[s0:s1], j[s0:s1]
        if wl.lat_fmt == LATENT_FP8:
            lat_v[p, jj] = e4m3_codes(x / tensor_scale)
        else:
            packed, sc = nvfp4_encode(x[:, :V_DIM].contiguous())
            codes_l[p, jj] = packed
            sc_l[p, jj] = sc
            rope_l[p, jj] = e4m3_codes(x[:, V_DIM:] / tensor_scale)

    # ---- queries
    R = wl.num_rows
    gq = _gen(device, wl.seed * 100 + 3)
    q_idx = e4m3_codes(torch.randn((R, IDX_HEADS, IDX_DIM), generator=gq, device=device))
    head_w = torch.rand((R, IDX_HEADS), generator=gq, device=device, dtype=torch.float32)
    q_mla = torch.randn((R, wl.heads, LAT_DIM), generator=gq, device=device).to(torch.bfloat16).view(torch.int16)

    return Inputs(
        wl=wl,
        idx_pool=idx_pool,
        lat_pool=lat_pool,
        tensor_scale=tensor_scale,
        block_table=torch.from_numpy(bt_np).to(device),
        row_req=torch.from_numpy(wl.row_req()).to(device),
        row_ctx=torch.from_numpy(wl.row_ctx()).to(device),
        q_idx=q_idx,
        head_w=head_w,
        q_mla=q_mla,
    )


def small_workload(name: str, ctx: list[int], rows_per_req: int = 1, rows_per_group: int = 1,
                   key_fmt: int = KEY_FP8, lat_fmt: int = LATENT_FP8, k: int = 2048, heads: int = 96,
                   seed: int = 7, extra_pages: float = 0.5) -> Workload:
    """An ad-hoc workload for tests (edge cases, ragged tails)."""
    return Workload(name, list(ctx), rows_per_req, rows_per_group, key_fmt, lat_fmt, k, heads, seed, extra_pages)


# ------------------------------------------------------------------ MSA
#
# The block-sparse variant (vLLM blog "Day-0 support for MiniMax-M3.1-Flash",
# section "MSA primer"): 128-token blocks, which are also the cache pages; one
# shared index-key head of 128 FP8 values per token (128 B, no scale); K and V
# of 4 KV heads x 128 dims in FP8 with one per-tensor scale each (1,024 B per
# token); one FP8 index query per GQA group; FP8 attention queries with one
# per-tensor scale (section "Blackwell-optimised MSA kernels": the queries stay
# FP8), heads_per_group of them per group.  Values are N(0,1) before encoding;
# per-tensor scales are amax / 448.

MSA_PAGE, MSA_DIM, MSA_GROUPS, MSA_BLOCKS = 128, 128, 4, 16
MSA_INDEX_PAGE_BYTES = MSA_PAGE * MSA_DIM
MSA_KV_PAGE_BYTES = MSA_GROUPS * 2 * MSA_PAGE * MSA_DIM


@dataclass
class MsaWorkload:
    name: str
    ctx: list[int]
    rows_per_req: int
    rows_per_group: int
    heads_per_group: int = 16
    seed: int = 0
    extra_pages: float = 0.25

    @property
    def num_rows(self) -> int:
        return len(self.ctx) * self.rows_per_req

    def row_ctx(self) -> np.ndarray:
        n = self.rows_per_req
        return np.asarray([L - n + 1 + i for L in self.ctx for i in range(n)], dtype=np.int32)

    def row_req(self) -> np.ndarray:
        return np.repeat(np.arange(len(self.ctx), dtype=np.int32), self.rows_per_req)


def msa_workload(name: str) -> MsaWorkload:
    if name == "msa_decode_tiny_4k":
        return MsaWorkload(name, [4096], 1, 1, seed=1100, extra_pages=1.0)
    if name == "msa_decode_b8_128k":
        return MsaWorkload(name, [131072] * 8, 1, 1, seed=1101)
    if name == "msa_verify_b4_64k":
        return MsaWorkload(name, [65536] * 4, 8, 8, seed=1102)
    if name == "msa_decode_b32_16k_64k":
        return MsaWorkload(name, _ctx_uniform(1103, 32, 16384, 65536), 1, 1, seed=1103)
    raise KeyError(name)


MSA_WORKLOADS = ("msa_decode_tiny_4k", "msa_decode_b8_128k", "msa_verify_b4_64k", "msa_decode_b32_16k_64k")


@dataclass
class MsaInputs:
    wl: MsaWorkload
    idx_pool: torch.Tensor        # uint8 [num_pages, 16384]
    kv_pool: torch.Tensor         # uint8 [num_pages, 131072]
    k_scale: float
    v_scale: float
    block_table: torch.Tensor     # int32 [B, max_pages] (128-token pages)
    row_req: torch.Tensor         # int32 [R]
    row_ctx: torch.Tensor         # int32 [R]
    q_idx: torch.Tensor           # uint8 [R, 4, 128] e4m3 codes
    q: torch.Tensor               # uint8 [R, 4 * heads_per_group, 128] e4m3 codes (times q_scale)
    q_scale: float

    @property
    def max_ctx(self) -> int:
        return max(self.wl.ctx)

    def np(self, name: str) -> np.ndarray:
        t = getattr(self, name)
        return t.cpu().numpy()

    def to(self, device) -> "MsaInputs":
        mv = {n: getattr(self, n).to(device) for n in
              ("idx_pool", "kv_pool", "block_table", "row_req", "row_ctx", "q_idx", "q")}
        return MsaInputs(self.wl, k_scale=self.k_scale, v_scale=self.v_scale, q_scale=self.q_scale, **mv)


def make_msa_inputs(wl: MsaWorkload, device="cpu", chunk_tokens: int = 1 << 16) -> MsaInputs:
    device = torch.device(device)
    bt_np, num_pages = _paging(wl, MSA_PAGE)
    slots = []
    for b, L in enumerate(wl.ctx):
        t = np.arange(L, dtype=np.int64)
        slots.append(bt_np[b, t // MSA_PAGE].astype(np.int64) * MSA_PAGE + t % MSA_PAGE)
    slots = torch.from_numpy(np.concatenate(slots)).to(device)
    T = slots.numel()
    pg, j = slots // MSA_PAGE, slots % MSA_PAGE

    idx_pool = torch.full((num_pages, MSA_INDEX_PAGE_BYTES), 0x7F, dtype=torch.uint8, device=device)
    idx_v = idx_pool.view(num_pages, MSA_PAGE, MSA_DIM)
    gk = _gen(device, wl.seed * 100 + 1)
    for s0 in range(0, T, chunk_tokens):
        s1 = min(T, s0 + chunk_tokens)
        idx_v[pg[s0:s1], j[s0:s1]] = e4m3_codes(torch.randn((s1 - s0, MSA_DIM), generator=gk, device=device))

    # K and V: per-tensor scale = amax / 448 over the used tokens (pass 1 records
    # amax, pass 2 redraws the same stream and encodes)
    kv_pool = torch.full((num_pages, MSA_KV_PAGE_BYTES), 0x7F, dtype=torch.uint8, device=device)
    kv_v = kv_pool.view(num_pages, MSA_GROUPS, 2, MSA_PAGE, MSA_DIM)
    amax = torch.zeros(2, device=device)
    gv = _gen(device, wl.seed * 100 + 2)
    for s0 in range(0, T, chunk_tokens):
        s1 = min(T, s0 + chunk_tokens)
        x = torch.randn((s1 - s0, MSA_GROUPS, 2, MSA_DIM), generator=gv, device=device)
        amax = torch.maximum(amax, x.abs().amax(dim=(0, 1, 3)))
    k_scale, v_scale = (float(a) / 448.0 if float(a) > 0 else 1.0 for a in amax.tolist())
    scale = torch.tensor([k_scale, v_scale], device=device).view(1, 1, 2, 1)
    gv = _gen(device, wl.seed * 100 + 2)
    for s0 in range(0, T, chunk_tokens):
        s1 = min(T, s0 + chunk_tokens)
        x = torch.randn((s1 - s0, MSA_GROUPS, 2, MSA_DIM), generator=gv, device=device)
        kv_v[pg[s0:s1], :, :, j[s0:s1]] = e4m3_codes(x / scale)

    R = wl.num_rows
    gq = _gen(device, wl.seed * 100 + 3)
    q_idx = e4m3_codes(torch.randn((R, MSA_GROUPS, MSA_DIM), generator=gq, device=device))
    x = torch.randn((R, MSA_GROUPS * wl.heads_per_group, MSA_DIM), generator=gq, device=device)
    am = float(x.abs().amax()) if x.numel() else 0.0
    q_scale = am / 448.0 if am > 0 else 1.0
    q = e4m3_codes(x / q_scale)
    return MsaInputs(wl, idx_pool, kv_pool, k_scale, v_scale, torch.from_numpy(bt_np).to(device),
                     torch.from_numpy(wl.row_req()).to(device), torch.from_numpy(wl.row_ctx()).to(device), q_idx, q,
                     q_scale)


def small_msa_workload(name: str, ctx: list[int], rows_per_req: int = 1, rows_per_group: int = 1,
                       heads_per_group: int = 16, seed: int = 7, extra_pages: float = 0.5) -> MsaWorkload:
    """An ad-hoc MSA workload for tests."""
    return MsaWorkload(name, list(ctx), rows_per_req, rows_per_group, heads_per_group, seed, extra_pages)
