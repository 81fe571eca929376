"""GPU parity of the batched variable-length E4M3 tail (gqa_attn_paged_e4m3_batch)
against the FP64 oracle, sequence by sequence.

Workload ("[Perf] Ship the qualified SM70 long-context layout and drop its
context fences", Changes): verifier tails of several sequences of different
lengths in one launch, with the context lengths read on the device so that a
captured graph replays as they grow.  Each sequence is a run of logical pages
of one shared E4M3 cache (one K and one V scale), reached through its own row
of the block-table matrix.  Envelope: max abs <= 1e-3, rel L2 <= 1e-2.
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


def _batch(ctxs, R, max_ctx, page=16, seed=0, Hq=6, Hkv=1):
    bi = inputs.paged_e4m3_batch_inputs(ctxs, R, max_ctx, seed=seed, page=page, Hq=Hq, Hkv=Hkv)
    return bi.cache, bi.tables, bi.q


def _run_and_check(cuda_lib, big, tables, q, ctxs, max_ctx, out=None, what=""):
    for b, ctx in enumerate(ctxs):
        ref = oracle.paged_e4m3(q[b], big.kcache, big.vcache, big.kscale, big.vscale, tables[b],
                                ctx, big.scale)
        _check(out[b], ref, f"{what} sequence {b} ctx={ctx}")


def _dev(big, tables, q, ctxs):
    dev = torch.device("cuda")
    ks = torch.tensor([big.kscale], dtype=torch.float32, device=dev)
    vs = torch.tensor([big.vscale], dtype=torch.float32, device=dev)
    return (q.to(dev), big.kcache.to(dev), big.vcache.to(dev), ks, vs, tables.to(dev),
            torch.tensor(ctxs, dtype=torch.int32, device=dev))


@pytest.mark.parametrize("R,ctxs", [
    (2, [5000, 300, 12000]),
    (8, [8, 129, 4096, 777]),
    (1, [20000, 1, 16, 17, 3000, 128]),
])
def test_batch_matches_oracle_per_sequence(cuda_lib, R, ctxs):
    ctxs = [max(c, R) for c in ctxs]
    max_ctx = max(ctxs)
    big, tables, q = _batch(ctxs, R, max_ctx, seed=len(ctxs) + R)
    qd, kc, vc, ks, vs, bt, cl = _dev(big, tables, q, ctxs)
    out = cuda_lib.paged_e4m3_batch(qd, kc, vc, ks, vs, bt, cl, max_ctx, big.scale)
    torch.cuda.synchronize()
    assert cuda_lib.device_error() == 0
    _run_and_check(cuda_lib, big, tables, q, ctxs, max_ctx, out.cpu(), f"R={R}")


@pytest.mark.parametrize("Hq,Hkv,R", [(6, 2, 4), (8, 1, 6), (6, 6, 3)])
def test_batch_other_groupings(cuda_lib, Hq, Hkv, R):
    ctxs = [3000, 70, 9000, 1]
    ctxs = [max(c, R) for c in ctxs]
    max_ctx = max(ctxs)
    big, tables, q = _batch(ctxs, R, max_ctx, seed=Hq + Hkv, Hq=Hq, Hkv=Hkv)
    qd, kc, vc, ks, vs, bt, cl = _dev(big, tables, q, ctxs)
    out = cuda_lib.paged_e4m3_batch(qd, kc, vc, ks, vs, bt, cl, max_ctx, big.scale)
    torch.cuda.synchronize()
    assert cuda_lib.device_error() == 0
    _run_and_check(cuda_lib, big, tables, q, ctxs, max_ctx, out.cpu(), f"Hq={Hq} Hkv={Hkv}")


def test_batch_graph_replay_with_changing_contexts(cuda_lib):
    R, max_ctx = 4, 9000
    ctxs = [9000, 100, 5000, 2500, 7777]
    big, tables, q = _batch(ctxs, R, max_ctx, seed=3)
    qd, kc, vc, ks, vs, bt, cl = _dev(big, tables, q, ctxs)
    out = torch.empty_like(qd)
    cuda_lib.paged_e4m3_batch(qd, kc, vc, ks, vs, bt, cl, max_ctx, big.scale, out=out)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cuda_lib.paged_e4m3_batch(qd, kc, vc, ks, vs, bt, cl, max_ctx, big.scale, out=out)
    for step in ([9000, 100, 5000, 2500, 7777], [4, 4, 4, 4, 4], [129, 8999, 300, 9000, 64],
                 [3000, 3001, 3002, 3003, 3004]):
        cl.copy_(torch.tensor(step, dtype=torch.int32))
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert cuda_lib.device_error() == 0
        _run_and_check(cuda_lib, big, tables, q, step, max_ctx, out.cpu(), f"replay {step}")


def test_batch_more_sequences_than_sms(cuda_lib):
    R = 1
    rng = np.random.default_rng(5)
    ctxs = [int(x) for x in rng.integers(1, 700, size=160)]
    max_ctx = 700
    big, tables, q = _batch(ctxs, R, max_ctx, seed=5)
    qd, kc, vc, ks, vs, bt, cl = _dev(big, tables, q, ctxs)
    out = cuda_lib.paged_e4m3_batch(qd, kc, vc, ks, vs, bt, cl, max_ctx, big.scale)
    torch.cuda.synchronize()
    assert cuda_lib.device_error() == 0
    _run_and_check(cuda_lib, big, tables, q, ctxs, max_ctx, out.cpu(), "160 sequences")


def test_batch_bitwise_reproducible_and_bad_context_flagged(cuda_lib):
    R, max_ctx = 2, 4000
    ctxs = [4000, 1000, 2000]
    big, tables, q = _batch(ctxs, R, max_ctx, seed=6)
    qd, kc, vc, ks, vs, bt, cl = _dev(big, tables, q, ctxs)
    a = cuda_lib.paged_e4m3_batch(qd, kc, vc, ks, vs, bt, cl, max_ctx, big.scale)
    b = cuda_lib.paged_e4m3_batch(qd, kc, vc, ks, vs, bt, cl, max_ctx, big.scale)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert cuda_lib.device_error() == 0
    cl.copy_(torch.tensor([4000, 99999, 2000], dtype=torch.int32))   # clamped to max_ctx
    c = cuda_lib.paged_e4m3_batch(qd, kc, vc, ks, vs, bt, cl, max_ctx, big.scale)
    torch.cuda.synchronize()
    assert cuda_lib.device_error() & cuda_lib.DEVERR_BAD_CTX_LEN
    _run_and_check(cuda_lib, big, tables, q, [4000, 4000, 2000], max_ctx, c.cpu(), "clamped")


def test_batch_head_size_128_matches_oracle(cuda_lib):
    """Batched variable-length tails at head size 128."""
    ctxs = [300, 5000, 12345, 64, 9000]
    R, max_ctx = 3, 16384
    bi = inputs.paged_e4m3_batch_inputs(ctxs, R, max_ctx, seed=128, D=128)
    c = bi.cache
    dev = torch.device("cuda")
    ks = torch.tensor([c.kscale], dtype=torch.float32, device=dev)
    vs = torch.tensor([c.vscale], dtype=torch.float32, device=dev)
    out = cuda_lib.paged_e4m3_batch(bi.q.to(dev), c.kcache.to(dev), c.vcache.to(dev), ks, vs,
                                    bi.tables.to(dev),
                                    torch.tensor(ctxs, dtype=torch.int32, device=dev), max_ctx,
                                    c.scale)
    torch.cuda.synchronize()
    assert cuda_lib.device_error() == 0
    for b, ctx in enumerate(ctxs):
        ref = oracle.paged_e4m3(bi.q[b], c.kcache, c.vcache, c.kscale, c.vscale, bi.tables[b],
                                ctx, c.scale)
        g = out[b].float().cpu().numpy().astype(np.float64)
        err = np.abs(g - ref).max()
        rel = np.linalg.norm(g - ref) / np.linalg.norm(ref)
        assert err <= 1e-3 and rel <= 1e-2, f"D=128 seq {b}: {err:.3e} {rel:.3e}"
