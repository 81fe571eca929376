"""GPU parity of the paged FP8-E4M3 verifier tail against the FP64 oracle.

Workload ("[Perf] Ship the qualified SM70 long-context layout and drop its
context fences", What / Changes / Measurement): R query rows (1..8) at the end
of a context up to the 262144 capacity, E4M3 K/V with one fp32 scale each in
page-16 blocks under a permuted block table.  Envelope: max abs <= 1e-3,
rel L2 <= 1e-2 ("[Kernel][SM70] Default long-prefill GQA architecture",
Test Result).
"""

import numpy as np
import pytest
import torch

import oracle
from long_context_causal_gqa_gb300 import inputs

pytestmark = pytest.mark.gpu


def _to_dev(p, dev):
    ks = torch.tensor([p.kscale], dtype=torch.float32, device=dev)
    vs = torch.tensor([p.vscale], dtype=torch.float32, device=dev)
    return (p.q.to(dev), p.kcache.to(dev), p.vcache.to(dev), ks, vs, p.block_table.to(dev))


def _check(got, ref, what):
    g = got.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(g).all(), what
    err = np.abs(g - ref).max()
    rel = np.linalg.norm(g - ref) / np.linalg.norm(ref)
    assert err <= 1e-3 and rel <= 1e-2, f"{what}: max abs {err:.3e} rel L2 {rel:.3e}"


def _run(lib, p):
    dev = torch.device("cuda")
    q, kc, vc, ks, vs, bt = _to_dev(p, dev)
    out = lib.paged_e4m3(q, kc, vc, ks, vs, bt, p.ctx_len, p.scale)
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    return out


@pytest.mark.parametrize("R,ctx,cap", [
    (1, 1, 16), (8, 8, 16), (1, 3000, 4096), (2, 3001, 4096), (8, 2999, 4096),
    (3, 130, 256), (5, 5000, 8192), (7, 1000, 1024), (4, 40000, 65536), (6, 777, 2048),
])
def test_paged_matches_oracle(cuda_lib, R, ctx, cap):
    p = inputs.paged_e4m3_inputs(R=R, ctx_len=ctx, capacity=cap, seed=R * 31 + ctx)
    out = _run(cuda_lib, p)
    ref = oracle.paged_e4m3(p.q, p.kcache, p.vcache, p.kscale, p.vscale, p.block_table,
                            p.ctx_len, p.scale)
    _check(out, ref, f"R={R} ctx={ctx}")


@pytest.mark.parametrize("Hq,Hkv,R,ctx,cap", [
    (6, 2, 8, 5000, 8192),    # three query heads per KV head: 24 packed rows, two launches
    (6, 3, 4, 3001, 4096),    # two per KV head
    (6, 6, 8, 2000, 2048),    # one per KV head: 8 packed rows, six launches
    (8, 1, 6, 4100, 8192),    # one KV head, 48 packed rows in one launch
    (4, 1, 3, 1500, 2048),
    (1, 1, 16, 2222, 4096),   # sixteen rows of a single head
    (12, 4, 5, 900, 1024),
    (8, 2, 2, 7000, 8192),
    (6, 2, 1, 1, 16),         # a one-token context
    (6, 3, 3, 130, 256),      # a ragged last tile
])
def test_paged_other_groupings_match_oracle(cuda_lib, Hq, Hkv, R, ctx, cap):
    p = inputs.paged_e4m3_inputs(R=R, ctx_len=ctx, capacity=cap, seed=Hq * 7 + Hkv + R,
                                 Hq=Hq, Hkv=Hkv)
    out = _run(cuda_lib, p)
    ref = oracle.paged_e4m3(p.q, p.kcache, p.vcache, p.kscale, p.vscale, p.block_table,
                            p.ctx_len, p.scale)
    _check(out, ref, f"Hq={Hq} Hkv={Hkv} R={R} ctx={ctx}")


@pytest.mark.parametrize("R", [1, 2, 8])
def test_paged_full_size(cuda_lib, R):
    p = inputs.paged_e4m3_inputs(R=R, ctx_len=261888, capacity=262144, seed=R)
    out = _run(cuda_lib, p)
    ref = oracle.paged_e4m3(p.q, p.kcache, p.vcache, p.kscale, p.vscale, p.block_table,
                            p.ctx_len, p.scale)
    _check(out, ref, f"R={R} ctx=261888")


def test_paged_bitwise_reproducible_and_graph_replay(cuda_lib):
    dev = torch.device("cuda")
    p = inputs.paged_e4m3_inputs(R=8, ctx_len=50000, capacity=65536, seed=11)
    q, kc, vc, ks, vs, bt = _to_dev(p, dev)
    a = cuda_lib.paged_e4m3(q, kc, vc, ks, vs, bt, p.ctx_len, p.scale)
    b = cuda_lib.paged_e4m3(q, kc, vc, ks, vs, bt, p.ctx_len, p.scale)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    out = torch.empty_like(q)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cuda_lib.paged_e4m3(q, kc, vc, ks, vs, bt, p.ctx_len, p.scale, out=out)
    for _ in range(2):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), a.view(torch.int16))
    assert cuda_lib.device_error() == 0


def test_paged_scale_is_read_on_device(cuda_lib):
    """Doubling vscale in device memory doubles the output (graph-capturable scales)."""
    dev = torch.device("cuda")
    p = inputs.paged_e4m3_inputs(R=2, ctx_len=4000, capacity=4096, seed=12)
    q, kc, vc, ks, vs, bt = _to_dev(p, dev)
    a = cuda_lib.paged_e4m3(q, kc, vc, ks, vs, bt, p.ctx_len, p.scale).float()
    vs.mul_(2.0)
    b = cuda_lib.paged_e4m3(q, kc, vc, ks, vs, bt, p.ctx_len, p.scale).float()
    torch.cuda.synchronize()
    assert torch.allclose(b, 2 * a, rtol=2e-3, atol=1e-6)


def test_paged_bad_page_id_sets_device_error(cuda_lib):
    dev = torch.device("cuda")
    p = inputs.paged_e4m3_inputs(R=1, ctx_len=500, capacity=512, seed=13)
    q, kc, vc, ks, vs, bt = _to_dev(p, dev)
    bt[3] = kc.shape[0] + 5
    cuda_lib.paged_e4m3(q, kc, vc, ks, vs, bt, p.ctx_len, p.scale)
    err = cuda_lib.device_error()
    assert err & cuda_lib.DEVERR_BAD_PAGE_ID
    assert cuda_lib.device_error() == 0  # read clears it


def _poison_past(kc_dev, vc_dev, bt, ctx_len, max_ctx):
    """Write the E4M3 NaN code into every cached token in [ctx_len, max_ctx)."""
    t = torch.arange(ctx_len, max_ctx)
    pg, slot = bt[t // 16].long(), t % 16
    kc_dev[pg, slot] = 0x7F
    vc_dev[pg, slot] = 0x7F


@pytest.mark.parametrize("R", [1, 5, 8])
def test_paged_devctx_graph_replay_at_growing_context(cuda_lib, R):
    """One graph captured at the bound, replayed with the context length
    changed on the device ([P2] Changes: tail graphs replayed as the context
    grows); tokens past each context are NaN-poisoned and must not matter."""
    max_ctx, cap = 9000, 9216
    p = inputs.paged_e4m3_inputs(R=R, ctx_len=max_ctx, capacity=cap, seed=40 + R)
    dev = torch.device("cuda")
    q, kc, vc, ks, vs, bt = _to_dev(p, dev)
    ctx_dev = torch.tensor([max_ctx], dtype=torch.int32, device=dev)
    out = torch.empty_like(q)
    cuda_lib.paged_e4m3_devctx(q, kc, vc, ks, vs, bt, ctx_dev, max_ctx, p.scale, out=out)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cuda_lib.paged_e4m3_devctx(q, kc, vc, ks, vs, bt, ctx_dev, max_ctx, p.scale, out=out)
    kc_host, vc_host = p.kcache.clone(), p.vcache.clone()
    for ctx in [max_ctx, 8999, 7000, 4097, 4096, 1000, 129, 128, 8 + R]:
        _poison_past(kc_host, vc_host, p.block_table, ctx, max_ctx)
        kc.copy_(kc_host)
        vc.copy_(vc_host)
        ctx_dev.fill_(ctx)
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert cuda_lib.device_error() == 0
        ref = oracle.paged_e4m3(p.q, kc_host, vc_host, p.kscale, p.vscale, p.block_table, ctx,
                                p.scale)
        _check(out, ref, f"R={R} device ctx={ctx}")


def test_paged_devctx_equals_host_ctx(cuda_lib):
    p = inputs.paged_e4m3_inputs(R=4, ctx_len=20000, capacity=20480, seed=77)
    dev = torch.device("cuda")
    q, kc, vc, ks, vs, bt = _to_dev(p, dev)
    a = cuda_lib.paged_e4m3(q, kc, vc, ks, vs, bt, p.ctx_len, p.scale)
    ctx_dev = torch.tensor([p.ctx_len], dtype=torch.int32, device=dev)
    b = cuda_lib.paged_e4m3_devctx(q, kc, vc, ks, vs, bt, ctx_dev, p.ctx_len, p.scale)
    torch.cuda.synchronize()
    # Same grid and split boundaries when max_ctx_len == ctx_len: bitwise equal.
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert cuda_lib.device_error() == 0


def test_paged_devctx_out_of_range_is_clamped_and_flagged(cuda_lib):
    p = inputs.paged_e4m3_inputs(R=2, ctx_len=3000, capacity=3072, seed=78)
    dev = torch.device("cuda")
    q, kc, vc, ks, vs, bt = _to_dev(p, dev)
    for bad, used in [(5000, 3000), (1, 2)]:
        ctx_dev = torch.tensor([bad], dtype=torch.int32, device=dev)
        out = cuda_lib.paged_e4m3_devctx(q, kc, vc, ks, vs, bt, ctx_dev, 3000, p.scale)
        torch.cuda.synchronize()
        assert cuda_lib.device_error() & cuda_lib.DEVERR_BAD_CTX_LEN
        if used == 3000:
            ref = oracle.paged_e4m3(p.q, p.kcache, p.vcache, p.kscale, p.vscale, p.block_table,
                                    used, p.scale)
            _check(out, ref, f"clamped ctx {bad} -> {used}")


@pytest.mark.parametrize("page,R,ctx,cap", [
    (8, 1, 3000, 4096), (8, 8, 777, 1024), (32, 2, 5001, 8192), (64, 5, 4000, 4096),
    (128, 8, 3333, 4096), (256, 3, 5000, 8192), (256, 1, 129, 256), (64, 8, 40000, 65536),
])
def test_paged_other_page_sizes(cuda_lib, page, R, ctx, cap):
    """Page sizes other than the pages' 16: a 128-key tile is TILE / page pages
    (page <= 128) or a slice of one page (page 256)."""
    p = inputs.paged_e4m3_inputs(R=R, ctx_len=ctx, capacity=cap, seed=page + R, page=page)
    out = _run(cuda_lib, p)
    ref = oracle.paged_e4m3(p.q, p.kcache, p.vcache, p.kscale, p.vscale, p.block_table,
                            p.ctx_len, p.scale)
    _check(out, ref, f"page={page} R={R} ctx={ctx}")


def test_paged_devctx_page_256_graph_replay(cuda_lib):
    max_ctx, cap = 6000, 6144
    p = inputs.paged_e4m3_inputs(R=4, ctx_len=max_ctx, capacity=cap, seed=91, page=256)
    dev = torch.device("cuda")
    q, kc, vc, ks, vs, bt = _to_dev(p, dev)
    ctx_dev = torch.tensor([max_ctx], dtype=torch.int32, device=dev)
    out = torch.empty_like(q)
    cuda_lib.paged_e4m3_devctx(q, kc, vc, ks, vs, bt, ctx_dev, max_ctx, p.scale, out=out)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cuda_lib.paged_e4m3_devctx(q, kc, vc, ks, vs, bt, ctx_dev, max_ctx, p.scale, out=out)
    for ctx in [6000, 3001, 256, 255, 100]:
        ctx_dev.fill_(ctx)
        g.replay()
        torch.cuda.synchronize()
        assert cuda_lib.device_error() == 0
        ref = oracle.paged_e4m3(p.q, p.kcache, p.vcache, p.kscale, p.vscale, p.block_table, ctx,
                                p.scale)
        _check(out, ref, f"page=256 device ctx={ctx}")


@pytest.mark.parametrize("Hq,Hkv,R,ctx,cap,page", [
    (6, 1, 1, 3000, 4096, 16),
    (6, 1, 8, 5000, 8192, 16),    # 48 packed rows
    (6, 1, 1, 1, 16, 16),         # a one-token context
    (6, 2, 8, 4000, 4096, 16),    # two launches of 24 packed rows
    (8, 1, 6, 3001, 4096, 32),
    (6, 3, 4, 777, 1024, 8),
    (4, 4, 5, 2000, 2048, 64),
    (6, 1, 8, 40000, 65536, 256),
    (6, 1, 3, 130, 256, 128),     # a ragged last tile
])
def test_paged_head_size_128_matches_oracle(cuda_lib, Hq, Hkv, R, ctx, cap, page):
    """Head size 128 (one 128-byte swizzle atom per cache row, 16 KB stages)."""
    p = inputs.paged_e4m3_inputs(R=R, ctx_len=ctx, capacity=cap, seed=Hq + R + page, page=page,
                                 Hq=Hq, Hkv=Hkv, D=128)
    out = _run(cuda_lib, p)
    _check(out, oracle.paged_e4m3(p.q, p.kcache, p.vcache, p.kscale, p.vscale, p.block_table,
                                  p.ctx_len, p.scale), f"D=128 Hq={Hq} Hkv={Hkv} R={R} ctx={ctx}")


@pytest.mark.parametrize("R", [1, 8])
def test_paged_head_size_128_full_size_and_replay(cuda_lib, R):
    p = inputs.paged_e4m3_inputs(R=R, ctx_len=261888, capacity=262144, seed=70 + R, D=128)
    dev = torch.device("cuda")
    q, kc, vc, ks, vs, bt = _to_dev(p, dev)
    a = cuda_lib.paged_e4m3(q, kc, vc, ks, vs, bt, p.ctx_len, p.scale)
    torch.cuda.synchronize()
    assert cuda_lib.device_error() == 0
    _check(a, oracle.paged_e4m3(p.q, p.kcache, p.vcache, p.kscale, p.vscale, p.block_table,
                                p.ctx_len, p.scale), f"D=128 R={R} ctx=261888")
    out = torch.empty_like(q)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cuda_lib.paged_e4m3(q, kc, vc, ks, vs, bt, p.ctx_len, p.scale, out=out)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), a.view(torch.int16))


def test_paged_head_size_128_devctx_replay(cuda_lib):
    max_ctx, cap = 9000, 9216
    p = inputs.paged_e4m3_inputs(R=4, ctx_len=max_ctx, capacity=cap, seed=93, D=128)
    dev = torch.device("cuda")
    q, kc, vc, ks, vs, bt = _to_dev(p, dev)
    ctx_dev = torch.tensor([max_ctx], dtype=torch.int32, device=dev)
    out = torch.empty_like(q)
    cuda_lib.paged_e4m3_devctx(q, kc, vc, ks, vs, bt, ctx_dev, max_ctx, p.scale, out=out)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cuda_lib.paged_e4m3_devctx(q, kc, vc, ks, vs, bt, ctx_dev, max_ctx, p.scale, out=out)
    for ctx in [9000, 4097, 128, 5]:
        ctx_dev.fill_(ctx)
        g.replay()
        torch.cuda.synchronize()
        assert cuda_lib.device_error() == 0
        ref = oracle.paged_e4m3(p.q, p.kcache, p.vcache, p.kscale, p.vscale, p.block_table, ctx,
                                p.scale)
        _check(out, ref, f"D=128 device ctx={ctx}")
