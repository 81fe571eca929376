"""GPU parity of the selected-block sparse prefill over an FP8-E4M3 page cache
(gqa_attn_sparse_blocks_e4m3) against the FP64 oracle.

Workload: the selections of "[Kernel][SM70] Repair #378 on latest main"
(Changes / Test Result) over the E4M3 storage of "[Perf] Ship the qualified
SM70 long-context layout and drop its context fences" (What): one fp32 scale
for K and one for V, unused pages and slots past the context holding the E4M3
NaN code.  Envelope: max abs <= 1e-3, rel L2 <= 1e-2; bitwise reproducible.
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


def _dev(s):
    dev = torch.device("cuda")
    ks = torch.tensor([s.kscale], dtype=torch.float32, device=dev)
    vs = torch.tensor([s.vscale], dtype=torch.float32, device=dev)
    return (s.q.to(dev), s.kcache.to(dev), s.vcache.to(dev), ks, vs, s.block_table.to(dev),
            s.sel_idx.to(dev), s.sel_cnt.to(dev))


def _run(lib, s, out=None):
    q, kc, vc, ks, vs, bt, si, sc = _dev(s)
    out = lib.sparse_blocks_e4m3(q, kc, vc, ks, vs, bt, si, sc, s.ctx_len, s.scale, out=out)
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    return out


def _ref(s, rows=None):
    return oracle.sparse_blocks_e4m3(s.q, s.kcache, s.vcache, s.kscale, s.vscale, s.block_table,
                                     s.sel_idx, s.sel_cnt, s.ctx_len, s.scale, rows=rows)


@pytest.mark.parametrize("rows,ctx,T,page", [
    (1, 4, 4, 16), (5, 41, 12, 16), (64, 2048, 64, 16), (100, 3001, 512, 16),
    (300, 5000, 200, 16), (200, 4096, 2048, 16), (77, 2000, 300, 8), (90, 3000, 256, 64),
    (77, 2000, 60, 8), (91, 3000, 64, 64), (33, 1500, 48, 256),
])
def test_sparse_e4m3_matches_oracle(cuda_lib, rows, ctx, T, page):
    s = inputs.sparse_e4m3_inputs(rows=rows, ctx_len=ctx, tokens=T, seed=rows + T, page=page,
                                  num_pages=(ctx + page - 1) // page + 3)
    _check(_run(cuda_lib, s), _ref(s), f"rows={rows} ctx={ctx} T={T} page={page}")


@pytest.mark.parametrize("Hq,Hkv,rows,ctx,T", [
    (6, 2, 100, 3001, 512), (8, 1, 120, 4096, 512), (6, 6, 50, 1500, 200), (16, 1, 40, 1000, 128),
])
def test_sparse_e4m3_other_groupings(cuda_lib, Hq, Hkv, rows, ctx, T):
    s = inputs.sparse_e4m3_inputs(rows=rows, ctx_len=ctx, tokens=T, seed=Hq * 3 + Hkv, Hq=Hq,
                                  Hkv=Hkv)
    _check(_run(cuda_lib, s), _ref(s), f"Hq={Hq} Hkv={Hkv}")


@pytest.mark.parametrize("T", [64, 512, 2048])
def test_sparse_e4m3_full_size_sampled_rows(cuda_lib, T):
    s = inputs.sparse_e4m3_inputs(rows=4096, ctx_len=32768, tokens=T, seed=T)
    out = _run(cuda_lib, s)
    rng = np.random.default_rng(T)
    rows = np.array(sorted(set([0, 1, 2, 3, 4095] + rng.choice(4096, 40, replace=False).tolist())),
                    dtype=np.int32)
    _check(out[torch.as_tensor(rows, dtype=torch.long)], _ref(s, rows=rows), f"T={T}")
    assert torch.isfinite(out.float()).all()


def test_sparse_e4m3_bitwise_reproducible_and_graph_replay(cuda_lib):
    s = inputs.sparse_e4m3_inputs(rows=500, ctx_len=8000, tokens=512, seed=9)
    q, kc, vc, ks, vs, bt, si, sc = _dev(s)
    a = cuda_lib.sparse_blocks_e4m3(q, kc, vc, ks, vs, bt, si, sc, s.ctx_len, s.scale)
    b = cuda_lib.sparse_blocks_e4m3(q, kc, vc, ks, vs, bt, si, sc, s.ctx_len, s.scale)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    out = torch.empty_like(q)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cuda_lib.sparse_blocks_e4m3(q, kc, vc, ks, vs, bt, si, sc, s.ctx_len, s.scale, out=out)
    for _ in range(2):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), a.view(torch.int16))
    assert cuda_lib.device_error() == 0


def test_sparse_e4m3_scales_are_read_on_the_device(cuda_lib):
    """Doubling the scale tensors' values (a graph replay reads them anew)
    matches the oracle at the doubled scales."""
    s = inputs.sparse_e4m3_inputs(rows=64, ctx_len=2048, tokens=256, seed=10)
    q, kc, vc, ks, vs, bt, si, sc = _dev(s)
    out = torch.empty_like(q)
    g = torch.cuda.CUDAGraph()
    cuda_lib.sparse_blocks_e4m3(q, kc, vc, ks, vs, bt, si, sc, s.ctx_len, s.scale, out=out)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        cuda_lib.sparse_blocks_e4m3(q, kc, vc, ks, vs, bt, si, sc, s.ctx_len, s.scale, out=out)
    ks.mul_(2.0)
    vs.mul_(0.5)
    g.replay()
    torch.cuda.synchronize()
    ref = oracle.sparse_blocks_e4m3(s.q, s.kcache, s.vcache, 2.0 * s.kscale, 0.5 * s.vscale,
                                    s.block_table, s.sel_idx, s.sel_cnt, s.ctx_len, s.scale)
    _check(out, ref, "scales x2 / x0.5")


def test_sparse_e4m3_empty_rows_and_bad_ids(cuda_lib):
    """400 rows (more than one row per CTA, so the copy pipeline runs across
    rows) with every third row selecting nothing: those rows are zero, the
    others match the oracle.  Then out-of-range ids: masked and flagged."""
    s = inputs.sparse_e4m3_inputs(rows=400, ctx_len=4000, tokens=64, seed=12)
    cnt0 = s.sel_cnt.clone()
    cnt0[::3] = 0
    s0 = inputs.SparseE4M3Inputs(**{**s.__dict__, "sel_cnt": cnt0})
    out = _run(cuda_lib, s0)
    empty = torch.arange(400)[::3]
    assert torch.count_nonzero(out[empty]) == 0
    keep = np.array([i for i in range(400) if i % 3], dtype=np.int32)
    _check(out[torch.as_tensor(keep, dtype=torch.long)], _ref(s0, rows=keep), "empty rows")
    # Out-of-range ids select nothing and flag an error; the result is unchanged.
    sel, cnt = s.sel_idx, s.sel_cnt
    wide = torch.full((400, sel.shape[1] + 2), -1, dtype=torch.int32)
    wide[:, : sel.shape[1]] = sel
    cntw = cnt.clone()
    for i in range(400):
        n = int(cnt[i])
        wide[i, n] = (4000 - 400 + i) // 4 + 5
        wide[i, n + 1] = -7
        cntw[i] = n + 2
    sw = inputs.SparseE4M3Inputs(**{**s.__dict__, "sel_idx": wide, "sel_cnt": cntw,
                                    "max_sel": wide.shape[1]})
    q, kc, vc, ks, vs, bt, si, sc = _dev(sw)
    outw = cuda_lib.sparse_blocks_e4m3(q, kc, vc, ks, vs, bt, si, sc, sw.ctx_len, sw.scale)
    torch.cuda.synchronize()
    assert cuda_lib.device_error() & cuda_lib.DEVERR_BAD_BLOCK_ID
    _check(outw, _ref(s), "with bad ids")
