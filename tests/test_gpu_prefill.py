"""GPU parity of the dense causal prefill against the FP64 oracle.

Pass criterion ("[Kernel][SM70] Default long-prefill GQA architecture", Test
Result): max abs error <= 1e-3 and relative L2 <= 1e-2, all outputs finite.
Output must also be bitwise reproducible across runs and CUDA-graph replay
("[Kernel][SM70] Repair #378 on latest main", Test Result: graph replay
bitwise equal to eager).
"""

import numpy as np
import pytest
import torch

import oracle
from long_context_causal_gqa_gb300 import inputs

pytestmark = pytest.mark.gpu

MAX_ABS = 1e-3
REL_L2 = 1e-2


def _check(got, ref, what=""):
    g = got.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(g).all(), what
    err = np.abs(g - ref).max()
    rel = np.linalg.norm(g - ref) / np.linalg.norm(ref)
    assert err <= MAX_ABS and rel <= REL_L2, f"{what}: max abs {err:.3e} rel L2 {rel:.3e}"
    return err, rel


def _run(lib, d):
    dev = torch.device("cuda")
    q, k, v = d.q.to(dev), d.k.to(dev), d.v.to(dev)
    out = lib.prefill(q, k, v, d.scale)
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    return out


@pytest.mark.parametrize("Q,KV", [
    (256, 1024),   # the small configuration, full comparison
    (1, 1),        # single key
    (1, 300),      # one row, many keys
    (7, 7),        # square causal
    (22, 150),     # one ragged q-tile (132 packed rows)
    (100, 333),    # several tiles, ragged KV tail
    (300, 300),    # square, many diagonal tiles
    (640, 2100),   # enough work to split q-tiles across CTAs
])
def test_prefill_matches_oracle(cuda_lib, Q, KV):
    d = inputs.dense_inputs(Q, KV, seed=Q + KV)
    out = _run(cuda_lib, d)
    ref = oracle.dense(d.q, d.k, d.v, d.scale)
    _check(out, ref, f"Q={Q} KV={KV}")


@pytest.mark.parametrize("Hq,Hkv,Q,KV", [
    (6, 2, 300, 1000),   # three query heads per KV head: one launch per query head
    (6, 3, 130, 700),    # two per KV head
    (6, 6, 257, 900),    # one per KV head (multi-head attention)
    (8, 2, 64, 400),
    (12, 4, 200, 650),
    (8, 1, 100, 777),    # one KV head, eight packed query heads
    (4, 1, 333, 1200),
    (1, 1, 513, 1500),   # one packed row per position
    (16, 1, 40, 90),     # 16 packed rows per position, 8 positions per 128-row tile
    (6, 2, 1, 1),        # one position, one key, six heads of the tile space
    (6, 3, 2, 700),
    (12, 4, 1, 33),
    (2, 2, 300, 301),    # multi-head attention, square-ish causal
])
def test_prefill_other_groupings_match_oracle(cuda_lib, Hq, Hkv, Q, KV):
    d = inputs.dense_inputs(Q, KV, seed=Q + KV + Hq, Hq=Hq, Hkv=Hkv)
    out = _run(cuda_lib, d)
    ref = oracle.dense(d.q, d.k, d.v, d.scale)
    _check(out, ref, f"Hq={Hq} Hkv={Hkv} Q={Q} KV={KV}")


@pytest.mark.parametrize("Hq,Hkv", [(6, 2), (8, 1)])
def test_prefill_groupings_split_and_replay(cuda_lib, Hq, Hkv):
    """Enough work per launch that pair tiles are cut between CTA pairs and
    merged; sampled rows against the oracle, then bitwise equality of a second
    run and of CUDA-graph replay (several launches per call when Hkv > 1)."""
    dev = torch.device("cuda")
    Q, KV = 2000, 9000
    d = inputs.dense_inputs(Q, KV, seed=11, Hq=Hq, Hkv=Hkv)
    q, k, v = d.q.to(dev), d.k.to(dev), d.v.to(dev)
    a = cuda_lib.prefill(q, k, v, d.scale)
    torch.cuda.synchronize()
    assert cuda_lib.device_error() == 0
    rows = _sample_rows(Q, n=24, seed=Hq)
    ref = oracle.dense(d.q, d.k, d.v, d.scale, rows=rows)
    _check(a[torch.as_tensor(rows, dtype=torch.long)], ref, f"Hq={Hq} Hkv={Hkv}")
    b = cuda_lib.prefill(q, k, v, d.scale)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    out = torch.empty_like(q)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        cuda_lib.prefill(q, k, v, d.scale, out=out)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cuda_lib.prefill(q, k, v, d.scale, out=out)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), a.view(torch.int16))
    assert cuda_lib.device_error() == 0


@pytest.mark.parametrize("Hq,Hkv,Q,KV", [
    (6, 1, 256, 1024),   # the small configuration at head size 128
    (6, 1, 1, 1),
    (6, 1, 22, 150),     # one ragged q-tile
    (6, 1, 300, 300),
    (8, 2, 100, 777),    # several KV heads: one launch, 3-D maps
    (4, 4, 257, 900),
])
def test_prefill_head_size_128_matches_oracle(cuda_lib, Hq, Hkv, Q, KV):
    d = inputs.dense_inputs(Q, KV, seed=Q + KV + 128, Hq=Hq, Hkv=Hkv, D=128)
    out = _run(cuda_lib, d)
    ref = oracle.dense(d.q, d.k, d.v, d.scale)
    _check(out, ref, f"D=128 Hq={Hq} Hkv={Hkv} Q={Q} KV={KV}")


@pytest.mark.parametrize("Hq,Hkv", [(6, 1), (6, 2)])
def test_prefill_head_size_128_split_and_replay(cuda_lib, Hq, Hkv):
    """Pair tiles cut between CTA pairs and merged, at head size 128; sampled
    rows against the oracle, bitwise equal on a second run and on graph replay."""
    dev = torch.device("cuda")
    Q, KV = 2000, 9000
    d = inputs.dense_inputs(Q, KV, seed=13, Hq=Hq, Hkv=Hkv, D=128)
    q, k, v = d.q.to(dev), d.k.to(dev), d.v.to(dev)
    a = cuda_lib.prefill(q, k, v, d.scale)
    torch.cuda.synchronize()
    assert cuda_lib.device_error() == 0
    rows = _sample_rows(Q, n=24, seed=Hq + 128)
    ref = oracle.dense(d.q, d.k, d.v, d.scale, rows=rows)
    _check(a[torch.as_tensor(rows, dtype=torch.long)], ref, f"D=128 Hq={Hq} Hkv={Hkv}")
    b = cuda_lib.prefill(q, k, v, d.scale)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    out = torch.empty_like(q)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cuda_lib.prefill(q, k, v, d.scale, out=out)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), a.view(torch.int16))


def _sample_rows(Q, n=48, seed=0):
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 20, 21, 22, 42, 43, Q // 2, Q - 22, Q - 2, Q - 1]
    rows = sorted(set([r for r in fixed if 0 <= r < Q] + rng.choice(Q, n, replace=False).tolist()))
    return np.array(rows, dtype=np.int32)


# The 12-shape sweep of "[Kernel][SM70] Default long-prefill GQA architecture"
# (Test Result: Q=8000, KV = 40000 .. 128000 in steps of 8000).
SWEEP_KV = list(range(40000, 128001, 8000))


@pytest.mark.parametrize("KV", SWEEP_KV)
def test_prefill_full_size_sampled_rows(cuda_lib, KV):
    Q = 8000
    d = inputs.dense_inputs(Q, KV, seed=1)
    out = _run(cuda_lib, d)
    rows = _sample_rows(Q, n=48 if KV in (40000, 128000) else 12, seed=KV)
    ref = oracle.dense(d.q, d.k, d.v, d.scale, rows=rows)
    _check(out[torch.as_tensor(rows, dtype=torch.long)], ref, f"Q={Q} KV={KV}")
    assert torch.isfinite(out.float()).all()


def test_prefill_bitwise_reproducible_and_graph_replay(cuda_lib):
    dev = torch.device("cuda")
    d = inputs.dense_inputs(700, 5000, seed=3)
    q, k, v = d.q.to(dev), d.k.to(dev), d.v.to(dev)
    a = cuda_lib.prefill(q, k, v, d.scale)
    b = cuda_lib.prefill(q, k, v, d.scale)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    out = torch.empty_like(q)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        cuda_lib.prefill(q, k, v, d.scale, out=out)  # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    out.zero_()
    with torch.cuda.graph(g):
        cuda_lib.prefill(q, k, v, d.scale, out=out)
    for _ in range(2):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), a.view(torch.int16))
    assert cuda_lib.device_error() == 0


# Changed future keys (row 0 bit-identical, every row against the oracle) and the
# other inputs that reach the softmax's rescale path: tests/test_gpu_edge.py.
