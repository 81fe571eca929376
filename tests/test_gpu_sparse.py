"""GPU parity of the selected-block sparse paged prefill against the FP64 oracle.

Workload ("[Kernel][SM70] Repair #378 on latest main", Changes / Test
Result): query rows at the end of an fp16 page-16 cache under a permuted
block table; each row attends its own selected four-token blocks, its own
block clamped to its position; tail counts 1/2/3 and non-monotonic tables are
among the page's cases.  Envelope: max abs <= 1e-3, rel L2 <= 1e-2.
"""

import numpy as np
import pytest
import torch

import oracle
from long_context_causal_gqa_gb300 import inputs

pytestmark = pytest.mark.gpu


def _check(got, ref, what):
    g = got.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(g).all(), what
    err = np.abs(g - ref).max()
    rel = np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-30)
    assert err <= 1e-3 and rel <= 1e-2, f"{what}: max abs {err:.3e} rel L2 {rel:.3e}"


def _dev(s, dev):
    return [x.to(dev) for x in (s.q, s.kcache, s.vcache, s.block_table, s.sel_idx, s.sel_cnt)]


def _run(lib, s, sel=None, cnt=None):
    dev = torch.device("cuda")
    q, kc, vc, bt, si, sc = _dev(s, dev)
    if sel is not None:
        si, sc = sel.to(dev), cnt.to(dev)
    out = lib.sparse_blocks(q, kc, vc, bt, si, sc, s.ctx_len, s.scale)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("rows,ctx,T", [
    (1, 4, 4), (5, 41, 12), (64, 2048, 64), (100, 3001, 512), (300, 5000, 200),
    (200, 4096, 2048),
])
def test_sparse_matches_oracle(cuda_lib, rows, ctx, T):
    s = inputs.sparse_inputs(rows=rows, ctx_len=ctx, tokens=T, seed=rows + T)
    out = _run(cuda_lib, s)
    assert cuda_lib.device_error() == 0
    ref = oracle.sparse_blocks(s.q, s.kcache, s.vcache, s.block_table, s.sel_idx, s.sel_cnt,
                               s.ctx_len, s.scale)
    _check(out, ref, f"rows={rows} ctx={ctx} T={T}")


@pytest.mark.parametrize("Hq,Hkv,rows,ctx,T", [
    (6, 2, 100, 3001, 512),   # three query heads per KV head, two launches
    (6, 3, 64, 2048, 64),
    (6, 6, 50, 1500, 200),    # one query head per KV head
    (8, 1, 120, 4096, 512),   # one KV head, eight query heads (generic instantiation)
    (16, 1, 40, 1000, 128),   # sixteen query heads: the full N granule
    (12, 4, 30, 900, 64),
    (4, 1, 77, 2000, 300),
    (1, 1, 90, 1200, 96),
    (6, 2, 1, 4, 4),          # one row, one block
    (6, 6, 5, 41, 12),
])
def test_sparse_other_groupings_match_oracle(cuda_lib, Hq, Hkv, rows, ctx, T):
    s = inputs.sparse_inputs(rows=rows, ctx_len=ctx, tokens=T, seed=Hq * 5 + Hkv, Hq=Hq, Hkv=Hkv)
    out = _run(cuda_lib, s)
    assert cuda_lib.device_error() == 0
    ref = oracle.sparse_blocks(s.q, s.kcache, s.vcache, s.block_table, s.sel_idx, s.sel_cnt,
                               s.ctx_len, s.scale)
    _check(out, ref, f"Hq={Hq} Hkv={Hkv} rows={rows} T={T}")


@pytest.mark.parametrize("T", [64, 512, 2048])
def test_sparse_full_size_sampled_rows(cuda_lib, T):
    s = inputs.sparse_inputs(rows=4096, ctx_len=32768, tokens=T, seed=T)
    out = _run(cuda_lib, s)
    assert cuda_lib.device_error() == 0
    rng = np.random.default_rng(T)
    rows = np.unique(np.concatenate([[0, 1, 2, 3, 4095], rng.choice(4096, 60, replace=False)]))
    ref = oracle.sparse_blocks(s.q, s.kcache, s.vcache, s.block_table, s.sel_idx, s.sel_cnt,
                               s.ctx_len, s.scale, rows=rows)
    _check(out[torch.as_tensor(rows, dtype=torch.long)], ref, f"T={T}")
    assert torch.isfinite(out.float()).all()


def test_sparse_every_block_equals_dense_prefill(cuda_lib):
    """Selecting every visible block of every row reproduces the dense kernel's math."""
    rows, ctx = 40, 700
    s = inputs.sparse_inputs(rows=rows, ctx_len=ctx, tokens=8, seed=5)
    nb = (ctx + 3) // 4
    sel = torch.full((rows, nb), -1, dtype=torch.int32)
    cnt = torch.zeros(rows, dtype=torch.int32)
    for i in range(rows):
        n = (ctx - rows + i) // 4 + 1
        sel[i, :n] = torch.arange(n, dtype=torch.int32)
        cnt[i] = n
    out = _run(cuda_lib, s, sel, cnt)
    n_log = (ctx + 15) // 16
    k = s.kcache[s.block_table[:n_log].long()].reshape(-1, 1, 256)[:ctx]
    v = s.vcache[s.block_table[:n_log].long()].reshape(-1, 1, 256)[:ctx]
    dense = cuda_lib.prefill(s.q.cuda(), k.contiguous().cuda(), v.contiguous().cuda(), s.scale)
    torch.cuda.synchronize()
    ref = oracle.dense(s.q, k, v, s.scale)
    _check(out, ref, "sparse(all blocks) vs oracle")
    _check(dense, ref, "dense vs oracle")


def test_sparse_tail_counts_and_bad_ids(cuda_lib):
    """Rows at p = 4b + {0,1,2,3} (tail counts 1..4), a row with no selection,
    and out-of-range ids (masked, flagged on the device)."""
    rows, ctx = 8, 1000
    s = inputs.sparse_inputs(rows=rows, ctx_len=ctx, tokens=40, seed=6)
    sel, cnt = s.sel_idx.clone(), s.sel_cnt.clone()
    out = _run(cuda_lib, s, sel, cnt)
    assert cuda_lib.device_error() == 0
    ref = oracle.sparse_blocks(s.q, s.kcache, s.vcache, s.block_table, sel, cnt, ctx, s.scale)
    _check(out, ref, "tail counts")
    # Row 2 selects nothing -> zero output.
    cnt0 = cnt.clone()
    cnt0[2] = 0
    out0 = _run(cuda_lib, s, sel, cnt0)
    assert cuda_lib.device_error() == 0
    assert torch.count_nonzero(out0[2]) == 0
    # Out-of-range ids select nothing and flag an error; the rest is unchanged.
    wide = torch.full((rows, sel.shape[1] + 2), -1, dtype=torch.int32)
    wide[:, : sel.shape[1]] = sel
    cntw = cnt.clone()
    for i in range(rows):
        n = int(cnt[i])
        wide[i, n] = (ctx - rows + i) // 4 + 5
        wide[i, n + 1] = -7
        cntw[i] = n + 2
    outw = _run(cuda_lib, s, wide, cntw)
    err = cuda_lib.device_error()
    assert err & cuda_lib.DEVERR_BAD_BLOCK_ID
    _check(outw, ref, "with bad ids")


def test_sparse_nan_poisoned_stale_tokens_do_not_leak(cuda_lib):
    """Tokens past the context are NaN in the generated cache; the last row's own
    block covers some of them, and they must be masked out."""
    s = inputs.sparse_inputs(rows=16, ctx_len=1003, tokens=64, seed=7)
    out = _run(cuda_lib, s)
    assert cuda_lib.device_error() == 0
    assert torch.isfinite(out.float()).all()


def test_sparse_bitwise_reproducible_and_graph_replay(cuda_lib):
    dev = torch.device("cuda")
    s = inputs.sparse_inputs(rows=512, ctx_len=8192, tokens=512, seed=8)
    args = _dev(s, dev)
    a = cuda_lib.sparse_blocks(*args, s.ctx_len, s.scale)
    b = cuda_lib.sparse_blocks(*args, s.ctx_len, s.scale)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    out = torch.empty_like(args[0])
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cuda_lib.sparse_blocks(*args, s.ctx_len, s.scale, out=out)
    for _ in range(2):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), a.view(torch.int16))
    assert cuda_lib.device_error() == 0


@pytest.mark.parametrize("page", [8, 32, 64, 256])
@pytest.mark.parametrize("T", [128, 60])
def test_sparse_other_page_sizes(cuda_lib, page, T):
    """Page sizes other than the pages' 16 (any power of two in [8, 256]);
    T = 60 (15 blocks per row) runs the two-rows-per-tile form, 97 rows the
    last unit with one row."""
    s = inputs.sparse_inputs(rows=97, ctx_len=3000, tokens=T, seed=page + T, page=page)
    out = _run(cuda_lib, s)
    ref = oracle.sparse_blocks(s.q, s.kcache, s.vcache, s.block_table, s.sel_idx, s.sel_cnt,
                               s.ctx_len, s.scale)
    _check(out, ref, f"page={page} T={T}")


def _with_duplicates(sel, cnt, seed, extra=8):
    """Each row's ids shuffled, then `extra` copies of randomly chosen ids of
    the row inserted at random positions (repeats within one 32-block tile
    and across tiles)."""
    g = torch.Generator().manual_seed(seed)
    rows = sel.shape[0]
    out = torch.full((rows, sel.shape[1] + extra), -1, dtype=torch.int32)
    cnt2 = cnt.clone()
    for i in range(rows):
        c = int(cnt[i])
        ids = sel[i, :c][torch.randperm(c, generator=g)]
        dups = ids[torch.randint(0, c, (extra,), generator=g)]
        allv = torch.cat([ids, dups])[torch.randperm(c + extra, generator=g)]
        out[i, : c + extra] = allv
        cnt2[i] = c + extra
    return out, cnt2


@pytest.mark.parametrize("ctx,e4m3,T,extra", [(4096, False, 512, 8), (4096, True, 512, 8),
                                              (70000, False, 512, 8), (4096, True, 40, 6),
                                              (4096, False, 40, 6)])
def test_sparse_duplicate_ids_are_masked_and_flagged(cuda_lib, ctx, e4m3, T, extra):
    """Selection has set semantics ("[Kernel][SM70] Repair #378 on latest
    main", Changes: stale or repeated entries are masked, not attended): a
    repeated id selects nothing more and sets GQA_DEVERR_DUP_BLOCK_ID.  Rows
    are shuffled and given repeats; the result equals the oracle's (which
    builds each row's visible set) and the error bit is set.  At ctx 70000
    the later rows' block ids exceed the kernel's exact 16384-bit set, so its
    hashed set with confirmation is exercised.  At T = 40 with 6 repeats (16
    positions) the kernels run two rows per tile and find repeats within
    each half of the tile."""
    rows = 301
    mk = inputs.sparse_e4m3_inputs if e4m3 else inputs.sparse_inputs
    s = mk(rows=rows, ctx_len=ctx, tokens=T, seed=31 + e4m3)
    sel, cnt = _with_duplicates(s.sel_idx, s.sel_cnt, seed=ctx + e4m3, extra=extra)
    dev = torch.device("cuda")
    if e4m3:
        ks = torch.tensor([s.kscale], dtype=torch.float32, device=dev)
        vs = torch.tensor([s.vscale], dtype=torch.float32, device=dev)
        out = cuda_lib.sparse_blocks_e4m3(s.q.to(dev), s.kcache.to(dev), s.vcache.to(dev), ks, vs,
                                          s.block_table.to(dev), sel.to(dev), cnt.to(dev),
                                          s.ctx_len, s.scale)
        ref = oracle.sparse_blocks_e4m3(s.q, s.kcache, s.vcache, s.kscale, s.vscale,
                                        s.block_table, sel, cnt, s.ctx_len, s.scale)
    else:
        out = _run(cuda_lib, s, sel, cnt)
        ref = oracle.sparse_blocks(s.q, s.kcache, s.vcache, s.block_table, sel, cnt, s.ctx_len,
                                   s.scale)
    torch.cuda.synchronize()
    err = cuda_lib.device_error()
    assert err & cuda_lib.DEVERR_DUP_BLOCK_ID
    assert not err & cuda_lib.DEVERR_BAD_BLOCK_ID
    _check(out, ref, f"duplicates ctx={ctx} e4m3={e4m3}")
    # Without repeats, shuffled ids give the same result within rounding and no error.
    sel1, cnt1 = _with_duplicates(s.sel_idx, s.sel_cnt, seed=7, extra=0)
    if not e4m3:
        out1 = _run(cuda_lib, s, sel1, cnt1)
        assert cuda_lib.device_error() == 0
        _check(out1, ref, "shuffled ids")


@pytest.mark.parametrize("Hq,Hkv,rows,ctx,T,page,e4m3", [
    (6, 1, 200, 4096, 512, 16, False),
    (6, 1, 200, 4096, 512, 16, True),
    (6, 1, 301, 4096, 64, 16, True),
    (6, 1, 301, 4096, 64, 16, False),
    (6, 1, 1, 4, 4, 16, False),          # one row, one block
    (6, 2, 100, 3001, 256, 32, False),   # two KV heads
    (8, 1, 120, 4096, 128, 8, True),     # generic 16-column instantiation
    (4, 4, 60, 2000, 64, 64, False),
    (6, 1, 300, 5000, 2048, 256, True),
    (16, 1, 40, 1000, 128, 16, False),
])
def test_sparse_head_size_128_matches_oracle(cuda_lib, Hq, Hkv, rows, ctx, T, page, e4m3):
    """Head size 128: a fp16 token row is 256 bytes (16 lanes, two keys per
    warp-wide copy), an E4M3 row 128 code bytes (8 lanes, four keys per pass)."""
    dev = torch.device("cuda")
    if e4m3:
        s = inputs.sparse_e4m3_inputs(rows=rows, ctx_len=ctx, tokens=T, seed=Hq + T, page=page,
                                      Hq=Hq, Hkv=Hkv, D=128)
        ks = torch.tensor([s.kscale], dtype=torch.float32, device=dev)
        vs = torch.tensor([s.vscale], dtype=torch.float32, device=dev)
        out = cuda_lib.sparse_blocks_e4m3(s.q.to(dev), s.kcache.to(dev), s.vcache.to(dev), ks, vs,
                                          s.block_table.to(dev), s.sel_idx.to(dev),
                                          s.sel_cnt.to(dev), s.ctx_len, s.scale)
        ref = oracle.sparse_blocks_e4m3(s.q, s.kcache, s.vcache, s.kscale, s.vscale,
                                        s.block_table, s.sel_idx, s.sel_cnt, s.ctx_len, s.scale)
    else:
        s = inputs.sparse_inputs(rows=rows, ctx_len=ctx, tokens=T, seed=Hq + T, page=page, Hq=Hq,
                                 Hkv=Hkv, D=128)
        out = _run(cuda_lib, s)
        ref = oracle.sparse_blocks(s.q, s.kcache, s.vcache, s.block_table, s.sel_idx, s.sel_cnt,
                                   s.ctx_len, s.scale)
    torch.cuda.synchronize()
    assert cuda_lib.device_error() == 0
    _check(out, ref, f"D=128 Hq={Hq} Hkv={Hkv} T={T} page={page} e4m3={e4m3}")


def test_sparse_head_size_128_full_size_sampled_rows(cuda_lib):
    s = inputs.sparse_inputs(rows=4096, ctx_len=32768, tokens=2048, seed=128, D=128)
    out = _run(cuda_lib, s)
    assert cuda_lib.device_error() == 0
    rows = np.array([0, 1, 2, 3, 1000, 2047, 4094, 4095], dtype=np.int32)
    ref = oracle.sparse_blocks(s.q, s.kcache, s.vcache, s.block_table, s.sel_idx, s.sel_cnt,
                               s.ctx_len, s.scale, rows=rows)
    _check(out[torch.as_tensor(rows, dtype=torch.long)], ref, "D=128 T=2048")
