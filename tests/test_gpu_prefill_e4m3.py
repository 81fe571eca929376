"""GPU parity of the dense causal prefill over an FP8-E4M3 K/V cache.

The E4M3 storage of "[Perf] Ship the qualified SM70 long-context layout and
drop its context fences" (What) applied to the dense workload of
"[Kernel][SM70] Default long-prefill GQA architecture" (Purpose): q fp16,
K and V E4M3 codes with one fp32 scale each.  Compared element by element with
the FP64 oracle over the same codes (max abs <= 1e-3, rel L2 <= 1e-2, the
pages' FP16 envelope), bitwise reproducible and equal under graph replay.
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


def _dev(d, dev):
    ks = torch.tensor([d.kscale], dtype=torch.float32, device=dev)
    vs = torch.tensor([d.vscale], dtype=torch.float32, device=dev)
    return d.q.to(dev), d.k.to(dev), d.v.to(dev), ks, vs


def _run(lib, d):
    out = lib.prefill_e4m3(*_dev(d, torch.device("cuda")), d.scale)
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    return out


# Every row sees at least ~100 keys: a row that sees one or a few keys outputs
# about one E4M3 value times the V scale, which fp16 holds only to half an ulp
# (up to 2^-9 at |v| >= 4, beyond the 1e-3 envelope; the fp16-input tests
# meet exact fp16 values there instead).
@pytest.mark.parametrize("Hq,Hkv,Q,KV,D", [
    (6, 1, 256, 1024, 256),   # the small configuration
    (6, 1, 1, 100, 256),      # one row
    (6, 1, 22, 150, 256),     # one ragged q-tile
    (6, 1, 300, 400, 256),    # many diagonal tiles
    (6, 1, 640, 2100, 256),   # pair tiles cut between CTA pairs
    (6, 2, 300, 1000, 256),   # two KV heads: every query head's tiles in one launch
    (8, 1, 100, 777, 256),
    (6, 1, 256, 1024, 128),   # head size 128
    (6, 1, 22, 150, 128),
    (8, 2, 100, 777, 128),
    (4, 4, 257, 900, 128),
])
def test_prefill_e4m3_matches_oracle(cuda_lib, Hq, Hkv, Q, KV, D):
    d = inputs.dense_e4m3_inputs(Q, KV, seed=Q + KV + D + Hq, Hq=Hq, Hkv=Hkv, D=D)
    out = _run(cuda_lib, d)
    ref = oracle.dense_e4m3(d.q, d.k, d.v, d.kscale, d.vscale, d.scale)
    _check(out, ref, f"E4M3 Hq={Hq} Hkv={Hkv} Q={Q} KV={KV} D={D}")


def _sample_rows(Q, n, seed):
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 20, 21, 22, 42, 43, Q // 2, Q - 22, Q - 2, Q - 1]
    rows = sorted(set([r for r in fixed if 0 <= r < Q] + rng.choice(Q, n, replace=False).tolist()))
    return np.array(rows, dtype=np.int32)


@pytest.mark.parametrize("Q,KV,D", [(8000, 40000, 256), (8000, 128000, 256), (8000, 40000, 128)])
def test_prefill_e4m3_full_size_sampled_rows(cuda_lib, Q, KV, D):
    d = inputs.dense_e4m3_inputs(Q, KV, seed=3, D=D)
    out = _run(cuda_lib, d)
    rows = _sample_rows(Q, 24, seed=KV + D)
    ref = oracle.dense_e4m3(d.q, d.k, d.v, d.kscale, d.vscale, d.scale, rows=rows)
    _check(out[torch.as_tensor(rows, dtype=torch.long)], ref, f"E4M3 Q={Q} KV={KV} D={D}")


@pytest.mark.parametrize("Hq,Hkv", [(6, 1), (6, 2)])
def test_prefill_e4m3_bitwise_reproducible_and_graph_replay(cuda_lib, Hq, Hkv):
    dev = torch.device("cuda")
    d = inputs.dense_e4m3_inputs(2000, 9000, seed=17, Hq=Hq, Hkv=Hkv)
    q, k, v, ks, vs = _dev(d, dev)
    a = cuda_lib.prefill_e4m3(q, k, v, ks, vs, d.scale)
    b = cuda_lib.prefill_e4m3(q, k, v, ks, vs, d.scale)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    rows = _sample_rows(2000, 16, seed=Hkv)
    ref = oracle.dense_e4m3(d.q, d.k, d.v, d.kscale, d.vscale, d.scale, rows=rows)
    _check(a[torch.as_tensor(rows, dtype=torch.long)], ref, f"E4M3 split Hq={Hq} Hkv={Hkv}")
    out = torch.empty_like(q)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cuda_lib.prefill_e4m3(q, k, v, ks, vs, d.scale, out=out)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), a.view(torch.int16))
    assert cuda_lib.device_error() == 0


def test_prefill_e4m3_scales_are_read_on_device(cuda_lib):
    """Doubling vscale in device memory doubles the output; doubling kscale
    equals halving the score scale (graph-capturable scales)."""
    dev = torch.device("cuda")
    d = inputs.dense_e4m3_inputs(300, 1000, seed=19)
    q, k, v, ks, vs = _dev(d, dev)
    a = cuda_lib.prefill_e4m3(q, k, v, ks, vs, d.scale).float()
    vs.mul_(2.0)
    b = cuda_lib.prefill_e4m3(q, k, v, ks, vs, d.scale).float()
    vs.div_(2.0)
    ks.mul_(2.0)
    c = cuda_lib.prefill_e4m3(q, k, v, ks, vs, d.scale / 2).float()
    torch.cuda.synchronize()
    assert torch.allclose(b, 2 * a, rtol=2e-3, atol=1e-6)
    assert torch.equal(c, a)


def test_prefill_e4m3_equals_fp16_prefill_on_decoded_values(cuda_lib):
    """At unit scales the E4M3 values are exact fp16 values: the fp16 prefill
    over the decoded cache runs the same UMMAs on the same operands, so the
    two kernels agree bit for bit."""
    dev = torch.device("cuda")
    d = inputs.dense_e4m3_inputs(640, 2100, seed=23)
    one = torch.ones(1, dtype=torch.float32, device=dev)
    a = cuda_lib.prefill_e4m3(d.q.to(dev), d.k.to(dev), d.v.to(dev), one, one, d.scale)
    k16 = d.k.view(torch.float8_e4m3fn).to(torch.float16).to(dev)
    v16 = d.v.view(torch.float8_e4m3fn).to(torch.float16).to(dev)
    b = cuda_lib.prefill(d.q.to(dev), k16, v16, d.scale)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
