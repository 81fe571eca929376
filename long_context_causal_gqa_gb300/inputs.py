"""Seeded synthetic inputs for the three attention workloads.

This module only draws and lays out input tensors (normal samples, an E4M3
encoding of them, permuted block tables, per-row block selections).  It holds
none of the attention arithmetic, so the CUDA path and the CPU oracle can both
be fed from it without sharing any of the method's code.

Workloads follow the pages "[Kernel][SM70] Default long-prefill GQA
architecture" (Purpose: Q=8000, KV=40000..128000, Hq=6, Hkv=1, D=256),
"[Perf] Ship the qualified SM70 long-context layout..." (What: grouped E4M3
long-context operator; Changes: capacity 262144, verifier tail) and
"[Kernel][SM70] Repair #378 on latest main" (Changes: selected four-token
blocks, page-16 caches in physical-page units).

Everything is generated on the CPU with ``torch.Generator().manual_seed(seed)``
and returned as CPU tensors; callers move them to the device.
"""

from __future__ import annotations

import dataclasses

import torch

HQ = 6
HKV = 1
HEAD_DIM = 256
SCALE = 1.0 / 16.0
PAGE = 16
SPARSE_BLOCK = 4
E4M3_MAX = 448.0
# Byte written into physical pages that no block-table entry points at.  0x7F
# is the E4M3 NaN code; a kernel that reads such a page produces wrong output.
E4M3_POISON = 0x7F


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(int(seed))
    return g


def normal_fp16(shape, seed: int) -> torch.Tensor:
    """i.i.d. N(0, 1) samples rounded to fp16."""
    return torch.randn(*shape, generator=_gen(seed), dtype=torch.float32).to(torch.float16)


@dataclasses.dataclass
class DenseInputs:
    q: torch.Tensor  # [Q, Hq, D] fp16
    k: torch.Tensor  # [KV, Hkv, D] fp16
    v: torch.Tensor  # [KV, Hkv, D] fp16
    Q: int
    KV: int
    Hq: int
    Hkv: int
    D: int
    scale: float


def dense_inputs(Q: int, KV: int, seed: int = 0, Hq: int = HQ, Hkv: int = HKV,
                 D: int = HEAD_DIM, scale: float = SCALE) -> DenseInputs:
    """Dense causal prefill inputs: q, k, v i.i.d. N(0,1) in fp16."""
    q = normal_fp16((Q, Hq, D), seed * 3 + 0)
    k = normal_fp16((KV, Hkv, D), seed * 3 + 1)
    v = normal_fp16((KV, Hkv, D), seed * 3 + 2)
    return DenseInputs(q, k, v, Q, KV, Hq, Hkv, D, scale)


@dataclasses.dataclass
class DenseE4M3Inputs:
    q: torch.Tensor  # [Q, Hq, D] fp16
    k: torch.Tensor  # [KV, Hkv, D] uint8 E4M3 codes
    v: torch.Tensor  # [KV, Hkv, D] uint8 E4M3 codes
    kscale: float
    vscale: float
    Q: int
    KV: int
    Hq: int
    Hkv: int
    D: int
    scale: float


def dense_e4m3_inputs(Q: int, KV: int, seed: int = 0, Hq: int = HQ, Hkv: int = HKV,
                      D: int = HEAD_DIM, scale: float = SCALE) -> "DenseE4M3Inputs":
    """Dense causal prefill over an E4M3 K/V cache: q i.i.d. N(0,1) in fp16; K and
    V i.i.d. N(0,1), each tensor encoded as E4M3 with one scale (absmax / 448),
    the storage of the E4M3 tail applied to the dense workload."""
    q = normal_fp16((Q, Hq, D), seed * 13 + 0)
    k, ks = e4m3_encode(torch.randn(KV, Hkv, D, generator=_gen(seed * 13 + 1)))
    v, vs = e4m3_encode(torch.randn(KV, Hkv, D, generator=_gen(seed * 13 + 2)))
    return DenseE4M3Inputs(q, k.contiguous(), v.contiguous(), ks, vs, Q, KV, Hq, Hkv, D, scale)


def e4m3_encode(x: torch.Tensor):
    """Per-tensor E4M3 encoding: scale = absmax / 448, byte = RNE(x / scale).

    Returns (bytes uint8 tensor of x's shape, fp32 scale).  Rounding is torch's
    float8_e4m3fn cast (round to nearest even); values are clamped to +-448
    first so no code saturates to NaN.
    """
    amax = float(x.abs().max()) if x.numel() else 1.0
    scale = amax / E4M3_MAX if amax > 0 else 1.0
    scale = float(torch.tensor(scale, dtype=torch.float32))
    y = (x.to(torch.float32) / scale).clamp_(-E4M3_MAX, E4M3_MAX)
    return y.to(torch.float8_e4m3fn).view(torch.uint8), scale


def permuted_block_table(num_logical: int, num_physical: int, seed: int) -> torch.Tensor:
    """Logical page n -> physical page id, a seeded random injection into
    ``range(num_physical)`` (the first ``num_logical`` entries of a permutation)."""
    perm = torch.randperm(num_physical, generator=_gen(seed))
    return perm[:num_logical].to(torch.int32).contiguous()


@dataclasses.dataclass
class PagedE4M3Inputs:
    q: torch.Tensor            # [R, Hq, D] fp16
    kcache: torch.Tensor       # [num_pages, page, Hkv, D] uint8 (E4M3 codes)
    vcache: torch.Tensor       # [num_pages, page, Hkv, D] uint8
    kscale: float
    vscale: float
    block_table: torch.Tensor  # [ceil(ctx_len / page)] int32 physical page ids
    ctx_len: int
    R: int
    page: int
    Hq: int
    Hkv: int
    D: int
    scale: float


def paged_e4m3_inputs(R: int, ctx_len: int, capacity: int = 262144, seed: int = 0,
                      page: int = PAGE, Hq: int = HQ, Hkv: int = HKV, D: int = HEAD_DIM,
                      scale: float = SCALE) -> PagedE4M3Inputs:
    """Paged FP8 verifier-tail inputs.

    K and V values for the ctx_len live tokens are N(0,1), encoded per tensor as
    E4M3 with one fp32 scale each.  Tokens are stored in page-``page`` blocks;
    the block table maps logical page n to a seeded random physical page out of
    ``capacity / page``; physical pages that no entry names hold the poison byte.
    """
    assert capacity % page == 0 and ctx_len <= capacity and 1 <= R <= ctx_len
    num_pages = capacity // page
    n_logical = (ctx_len + page - 1) // page
    q = normal_fp16((R, Hq, D), seed * 5 + 0)
    kv_vals = []
    for i in (1, 2):
        x = torch.randn(ctx_len, Hkv, D, generator=_gen(seed * 5 + i), dtype=torch.float32)
        kv_vals.append(x)
    kb, kscale = e4m3_encode(kv_vals[0])
    vb, vscale = e4m3_encode(kv_vals[1])
    table = permuted_block_table(n_logical, num_pages, seed * 5 + 3)
    caches = []
    for b in (kb, vb):
        cache = torch.full((num_pages, page, Hkv, D), E4M3_POISON, dtype=torch.uint8)
        padded = torch.full((n_logical * page, Hkv, D), E4M3_POISON, dtype=torch.uint8)
        padded[:ctx_len] = b
        cache[table.long()] = padded.view(n_logical, page, Hkv, D)
        caches.append(cache)
    return PagedE4M3Inputs(q, caches[0], caches[1], kscale, vscale, table, ctx_len, R,
                           page, Hq, Hkv, D, scale)


@dataclasses.dataclass
class PagedE4M3BatchInputs:
    cache: PagedE4M3Inputs     # the shared cache, scales and its own (unused) tail q
    tables: torch.Tensor       # [batch, stride] int32: sequence b's logical pages
    q: torch.Tensor            # [batch, R, Hq, D] fp16
    ctx_lens: list             # per-sequence context lengths
    max_ctx: int


def paged_e4m3_batch_inputs(ctx_lens, R: int, max_ctx: int, seed: int = 0, page: int = PAGE,
                            Hq: int = HQ, Hkv: int = HKV, D: int = HEAD_DIM,
                            scale: float = SCALE) -> PagedE4M3BatchInputs:
    """Batched verifier tails over one shared E4M3 cache: sequence b owns a run
    of ceil(max_ctx / page) consecutive logical pages of one permuted cache
    (the whole run is addressable, so its context can grow up to max_ctx),
    reached through row b of the block-table matrix; q per sequence is N(0,1)
    fp16.  Physical pages that no sequence names hold the poison byte."""
    assert all(1 <= R <= c <= max_ctx for c in ctx_lens)
    per = (max_ctx + page - 1) // page
    total = per * len(ctx_lens) * page
    cache = paged_e4m3_inputs(R=1, ctx_len=total, capacity=total + 4 * page, seed=seed,
                              page=page, Hq=Hq, Hkv=Hkv, D=D, scale=scale)
    tables = cache.block_table[: per * len(ctx_lens)].view(len(ctx_lens), per).clone()
    q = normal_fp16((len(ctx_lens), R, Hq, D), seed * 5 + 4)
    return PagedE4M3BatchInputs(cache, tables, q, list(ctx_lens), max_ctx)


@dataclasses.dataclass
class SparseInputs:
    q: torch.Tensor            # [rows, Hq, D] fp16
    kcache: torch.Tensor       # [num_pages, page, Hkv, D] fp16
    vcache: torch.Tensor       # [num_pages, page, Hkv, D] fp16
    block_table: torch.Tensor  # [ceil(ctx_len / page)] int32
    sel_idx: torch.Tensor      # [rows, max_sel] int32 logical 4-token block ids (-1 padding)
    sel_cnt: torch.Tensor      # [rows] int32
    max_sel: int
    ctx_len: int
    rows: int
    page: int
    Hq: int
    Hkv: int
    D: int
    scale: float


def sparse_selection(rows: int, ctx_len: int, tokens: int, seed: int,
                     block: int = SPARSE_BLOCK):
    """Per-row selections of ``tokens / block`` distinct causally visible blocks.

    Row i sits at position p = ctx_len - rows + i.  Its own (possibly partial)
    block p // block is always selected; the other blocks are drawn uniformly
    without replacement from 0 .. p // block - 1 (fewer if the row has fewer).
    Entries are ascending; unused tail entries are -1.
    """
    want = max(1, tokens // block)
    pos = torch.arange(rows, dtype=torch.int64) + (ctx_len - rows)
    own = pos // block
    nb = int(own.max()) + 1
    g = _gen(seed)
    keys = torch.rand(rows, nb, generator=g)
    ids = torch.arange(nb, dtype=torch.int64).unsqueeze(0)
    keys = torch.where(ids < own.unsqueeze(1), keys, torch.full_like(keys, 2.0))
    n_other = torch.clamp(own, max=want - 1)
    max_sel = want
    sel = torch.full((rows, max_sel), -1, dtype=torch.int64)
    if want > 1:
        _, idx = torch.topk(keys, want - 1, dim=1, largest=False, sorted=True)
        # Keep only the first n_other picks of each row (the rest landed on ids >= own).
        take = torch.arange(want - 1).unsqueeze(0) < n_other.unsqueeze(1)
        picked = torch.where(take, idx, torch.full_like(idx, 1 << 40))
        picked, _ = torch.sort(picked, dim=1)
        sel[:, : want - 1] = torch.where(picked < (1 << 40), picked, torch.full_like(picked, -1))
    cnt = n_other + 1
    # Place the own block right after the other picks; keep each row ascending.
    rows_idx = torch.arange(rows)
    sel[rows_idx, n_other] = own
    return sel.to(torch.int32).contiguous(), cnt.to(torch.int32).contiguous(), max_sel


def sparse_inputs(rows: int, ctx_len: int, tokens: int, seed: int = 0, page: int = PAGE,
                  Hq: int = HQ, Hkv: int = HKV, D: int = HEAD_DIM, scale: float = SCALE,
                  num_pages: int | None = None) -> SparseInputs:
    """Selected-block sparse paged prefill inputs (fp16 cache, N(0,1) values)."""
    assert 1 <= rows <= ctx_len
    n_logical = (ctx_len + page - 1) // page
    if num_pages is None:
        num_pages = n_logical
    q = normal_fp16((rows, Hq, D), seed * 7 + 0)
    table = permuted_block_table(n_logical, num_pages, seed * 7 + 3)
    caches = []
    for i in (1, 2):
        x = normal_fp16((n_logical * page, Hkv, D), seed * 7 + i)
        x[ctx_len:] = float("nan")
        cache = torch.full((num_pages, page, Hkv, D), float("nan"), dtype=torch.float16)
        cache[table.long()] = x.view(n_logical, page, Hkv, D)
        caches.append(cache)
    sel, cnt, max_sel = sparse_selection(rows, ctx_len, tokens, seed * 7 + 4)
    return SparseInputs(q, caches[0], caches[1], table, sel, cnt, max_sel, ctx_len, rows,
                        page, Hq, Hkv, D, scale)



@dataclasses.dataclass
class SparseE4M3Inputs:
    q: torch.Tensor            # [rows, Hq, D] fp16
    kcache: torch.Tensor       # [num_pages, page, Hkv, D] uint8 E4M3 codes
    vcache: torch.Tensor       # [num_pages, page, Hkv, D] uint8 E4M3 codes
    kscale: float
    vscale: float
    block_table: torch.Tensor  # [ceil(ctx_len / page)] int32
    sel_idx: torch.Tensor      # [rows, max_sel] int32 logical 4-token block ids (-1 padding)
    sel_cnt: torch.Tensor      # [rows] int32
    max_sel: int
    ctx_len: int
    rows: int
    page: int
    Hq: int
    Hkv: int
    D: int
    scale: float


def sparse_e4m3_inputs(rows: int, ctx_len: int, tokens: int, seed: int = 0, page: int = PAGE,
                       Hq: int = HQ, Hkv: int = HKV, D: int = HEAD_DIM, scale: float = SCALE,
                       num_pages: int | None = None) -> SparseE4M3Inputs:
    """Selected-block sparse inputs over an E4M3 page cache: q, block table and
    selections as in ``sparse_inputs``; K and V N(0,1) for the ctx_len live
    tokens, encoded per tensor as E4M3 with one fp32 scale each (absmax / 448,
    as the tail's cache); physical pages that no entry names, and slots past
    ctx_len, hold the poison byte."""
    assert 1 <= rows <= ctx_len
    n_logical = (ctx_len + page - 1) // page
    if num_pages is None:
        num_pages = n_logical
    q = normal_fp16((rows, Hq, D), seed * 11 + 0)
    table = permuted_block_table(n_logical, num_pages, seed * 11 + 3)
    caches, scales = [], []
    for i in (1, 2):
        x = torch.randn(ctx_len, Hkv, D, generator=_gen(seed * 11 + i), dtype=torch.float32)
        b, sc = e4m3_encode(x)
        padded = torch.full((n_logical * page, Hkv, D), E4M3_POISON, dtype=torch.uint8)
        padded[:ctx_len] = b
        cache = torch.full((num_pages, page, Hkv, D), E4M3_POISON, dtype=torch.uint8)
        cache[table.long()] = padded.view(n_logical, page, Hkv, D)
        caches.append(cache)
        scales.append(sc)
    sel, cnt, max_sel = sparse_selection(rows, ctx_len, tokens, seed * 11 + 4)
    return SparseE4M3Inputs(q, caches[0], caches[1], scales[0], scales[1], table, sel, cnt,
                            max_sel, ctx_len, rows, page, Hq, Hkv, D, scale)


def paged_e4m3_from_values(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, capacity: int,
                           seed: int = 0, page: int = PAGE,
                           scale: float = SCALE) -> PagedE4M3Inputs:
    """Paged E4M3 tail inputs laid out from given values: q [R, Hq, D] fp16,
    k / v [ctx_len, Hkv, D] real values, each tensor encoded as E4M3 with one
    scale (absmax / 448) and stored in page-``page`` blocks under a seeded
    permuted block table; unnamed pages and slots past ctx_len hold the poison
    byte.  Used for structured inputs (ramps, dominant keys, constant values)."""
    ctx_len, Hkv, D = k.shape
    R, Hq, _ = q.shape
    assert capacity % page == 0 and ctx_len <= capacity and 1 <= R <= ctx_len
    num_pages = capacity // page
    n_logical = (ctx_len + page - 1) // page
    table = permuted_block_table(n_logical, num_pages, seed * 5 + 3)
    caches, scales = [], []
    for x in (k, v):
        b, sc = e4m3_encode(x.to(torch.float32))
        cache = torch.full((num_pages, page, Hkv, D), E4M3_POISON, dtype=torch.uint8)
        padded = torch.full((n_logical * page, Hkv, D), E4M3_POISON, dtype=torch.uint8)
        padded[:ctx_len] = b
        cache[table.long()] = padded.view(n_logical, page, Hkv, D)
        caches.append(cache)
        scales.append(sc)
    return PagedE4M3Inputs(q.to(torch.float16).contiguous(), caches[0], caches[1], scales[0],
                           scales[1], table, ctx_len, R, page, Hq, Hkv, D, scale)


def sparse_from_values(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, tokens: int,
                       seed: int = 0, page: int = PAGE, scale: float = SCALE,
                       e4m3: bool = False):
    """Selected-block sparse inputs laid out from given values: q [rows, Hq, D],
    k / v [ctx_len, Hkv, D]; an fp16 cache (or, with e4m3, E4M3 codes with one
    scale per tensor) in a seeded permuted page table, NaN / poison past
    ctx_len and in unnamed pages, and seeded selections as ``sparse_inputs``."""
    ctx_len, Hkv, D = k.shape
    rows, Hq, _ = q.shape
    assert 1 <= rows <= ctx_len
    n_logical = (ctx_len + page - 1) // page
    num_pages = n_logical
    table = permuted_block_table(n_logical, num_pages, seed * 7 + 3)
    caches, scales = [], []
    for x in (k, v):
        if e4m3:
            b, sc = e4m3_encode(x.to(torch.float32))
            padded = torch.full((n_logical * page, Hkv, D), E4M3_POISON, dtype=torch.uint8)
            padded[:ctx_len] = b
            cache = torch.full((num_pages, page, Hkv, D), E4M3_POISON, dtype=torch.uint8)
            scales.append(sc)
        else:
            padded = torch.full((n_logical * page, Hkv, D), float("nan"), dtype=torch.float16)
            padded[:ctx_len] = x.to(torch.float16)
            cache = torch.full((num_pages, page, Hkv, D), float("nan"), dtype=torch.float16)
        cache[table.long()] = padded.view(n_logical, page, Hkv, D)
        caches.append(cache)
    sel, cnt, max_sel = sparse_selection(rows, ctx_len, tokens, seed * 7 + 4)
    qh = q.to(torch.float16).contiguous()
    if e4m3:
        return SparseE4M3Inputs(qh, caches[0], caches[1], scales[0], scales[1], table, sel, cnt,
                                max_sel, ctx_len, rows, page, Hq, Hkv, D, scale)
    return SparseInputs(qh, caches[0], caches[1], table, sel, cnt, max_sel, ctx_len, rows, page,
                        Hq, Hkv, D, scale)
