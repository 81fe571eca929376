"""Cache layouts of "[Kernel][SM70] Repair #378 on latest main" (Test Result)
served through the existing C ABI, checked on the GPU against the FP64 oracle.

* Interleaved K/V: one cache tensor [pages, 2, page, Hkv, D] holding page p's
  K block and then its V block.  Seen as 2 * pages blocks of one page each, K
  of logical page n is block 2 * table[n] and V is block 2 * table[n] + 1, so
  the call takes kcache = block 0, vcache = block 1 (both views of 2 * pages -
  1 blocks) and a table with every entry doubled.  The result must be bitwise
  equal to the same data in separate K and V caches.
* Hybrid 784/16 geometry: physical pages of 784 tokens addressed through a
  page-16 table; a 784-token page is 49 consecutive 16-token blocks, so the
  cache is read as page 16 with a non-monotonic 128-entry table.
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
    rel = np.linalg.norm(g - ref) / np.linalg.norm(ref)
    assert err <= 1e-3 and rel <= 1e-2, f"{what}: max abs {err:.3e} rel L2 {rel:.3e}"


def _interleave(kcache, vcache, table):
    """[pages, page, Hkv, D] K and V -> views of one interleaved cache, and the
    doubled table."""
    both = torch.stack([kcache, vcache], dim=1).contiguous()   # [pages, 2, page, Hkv, D]
    pages = kcache.shape[0]
    blocks = both.view(2 * pages, *kcache.shape[1:])
    return both, blocks[: 2 * pages - 1], blocks[1:], (table * 2).to(torch.int32)


@pytest.mark.parametrize("R,ctx,cap", [(1, 3000, 4096), (8, 9001, 16384)])
def test_paged_interleaved_kv(cuda_lib, R, ctx, cap):
    dev = torch.device("cuda")
    p = inputs.paged_e4m3_inputs(R=R, ctx_len=ctx, capacity=cap, seed=70 + R)
    ks = torch.tensor([p.kscale], dtype=torch.float32, device=dev)
    vs = torch.tensor([p.vscale], dtype=torch.float32, device=dev)
    q = p.q.to(dev)
    sep = cuda_lib.paged_e4m3(q, p.kcache.to(dev), p.vcache.to(dev), ks, vs,
                              p.block_table.to(dev), ctx, p.scale)
    both, kview, vview, table2 = _interleave(p.kcache, p.vcache, p.block_table)
    both = both.to(dev)
    blocks = both.view(2 * p.kcache.shape[0], *p.kcache.shape[1:])
    out = cuda_lib.paged_e4m3(q, blocks[:-1], blocks[1:], ks, vs, table2.to(dev), ctx, p.scale)
    torch.cuda.synchronize()
    assert cuda_lib.device_error() == 0
    assert torch.equal(out.view(torch.int16), sep.view(torch.int16))
    ref = oracle.paged_e4m3(p.q, kview, vview, p.kscale, p.vscale, table2, ctx, p.scale)
    _check(out, ref, f"interleaved R={R}")


def test_sparse_interleaved_kv(cuda_lib):
    dev = torch.device("cuda")
    s = inputs.sparse_inputs(rows=300, ctx_len=4096, tokens=512, seed=71)
    both, kview, vview, table2 = _interleave(s.kcache, s.vcache, s.block_table)
    both = both.to(dev)
    blocks = both.view(2 * s.kcache.shape[0], *s.kcache.shape[1:])
    q, si, sc = s.q.to(dev), s.sel_idx.to(dev), s.sel_cnt.to(dev)
    sep = cuda_lib.sparse_blocks(q, s.kcache.to(dev), s.vcache.to(dev), s.block_table.to(dev),
                                 si, sc, s.ctx_len, s.scale)
    out = cuda_lib.sparse_blocks(q, blocks[:-1], blocks[1:], table2.to(dev), si, sc, s.ctx_len,
                                 s.scale)
    torch.cuda.synchronize()
    assert cuda_lib.device_error() == 0
    assert torch.equal(out.view(torch.int16), sep.view(torch.int16))
    ref = oracle.sparse_blocks(s.q, kview, vview, table2, s.sel_idx, s.sel_cnt, s.ctx_len,
                               s.scale)
    _check(out, ref, "sparse interleaved")


def test_sparse_hybrid_784_16_geometry(cuda_lib):
    dev = torch.device("cuda")
    big_pages, big = 3, 784
    # 128 logical page-16 blocks (2048 tokens) spread over the 147 16-token
    # blocks of three 784-token pages by a seeded permutation.
    s = inputs.sparse_inputs(rows=256, ctx_len=2048, tokens=64, seed=72,
                             num_pages=big_pages * big // 16)
    table = s.block_table
    assert table.numel() == 128 and not bool((table[1:] > table[:-1]).all())
    k784 = s.kcache.reshape(big_pages, big, *s.kcache.shape[2:])   # the physical layout
    v784 = s.vcache.reshape(big_pages, big, *s.vcache.shape[2:])
    k16 = k784.to(dev).view(-1, 16, *s.kcache.shape[2:])
    v16 = v784.to(dev).view(-1, 16, *s.vcache.shape[2:])
    out = cuda_lib.sparse_blocks(s.q.to(dev), k16, v16, table.to(dev), s.sel_idx.to(dev),
                                 s.sel_cnt.to(dev), s.ctx_len, s.scale)
    torch.cuda.synchronize()
    assert cuda_lib.device_error() == 0
    ref = oracle.sparse_blocks(s.q, s.kcache, s.vcache, table, s.sel_idx, s.sel_cnt, s.ctx_len,
                               s.scale)
    _check(out, ref, "hybrid 784/16")
