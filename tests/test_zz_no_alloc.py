"""The allocation-free paged E4M3 entry point against the workspace-based one.

gqa_attn_paged_e4m3_noalloc serves callers that cannot call cudaMalloc (a
pooling allocator owns device memory, an allocation's implicit device
synchronisation is not acceptable in a serving loop, or plugin code has no
allocator).  It keeps its split partials in a static device array inside the
library instead of a registered workspace.  This test calls it through the C
ABI twice in a row and checks each result against gqa_attn_paged_e4m3 within
the tolerance the other GPU tests use (max abs 1e-3, relative L2 1e-2), for
bitwise equality where both run the same split partition (devices with at
most 160 SMs), and, at 1 and 8 rows, against the FP64 oracle.  It
lives in its own file, collected last, and passes alone in a fresh process as
well as after the other tests.
"""

import ctypes

import numpy as np
import pytest
import torch

from long_context_causal_gqa_gb300 import binding, inputs

pytestmark = pytest.mark.gpu


def _close_to_oracle(got, ref):
    g = got.float().cpu().numpy().astype(np.float64)
    err = np.abs(g - ref).max()
    rel = np.linalg.norm(g - ref) / np.linalg.norm(ref)
    assert err <= 1e-3 and rel <= 1e-2, f"vs oracle: max abs {err:.3e} rel L2 {rel:.3e}"


def _close(got, ref):
    g = got.float().cpu().numpy().astype(np.float64)
    r = ref.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(g).all()
    err = np.abs(g - r).max()
    rel = np.linalg.norm(g - r) / np.linalg.norm(r)
    assert err <= 1e-3 and rel <= 1e-2, f"max abs {err:.3e} rel L2 {rel:.3e}"


@pytest.mark.parametrize("R", [8, 2, 1])
def test_noalloc_matches_workspace_entry_point_twice(cuda_lib, R):
    dev = torch.device("cuda")
    p = inputs.paged_e4m3_inputs(R=R, ctx_len=30001, capacity=32768, seed=40 + R)
    q, kc, vc, bt = p.q.to(dev), p.kcache.to(dev), p.vcache.to(dev), p.block_table.to(dev)
    ks = torch.tensor([p.kscale], dtype=torch.float32, device=dev)
    vs = torch.tensor([p.vscale], dtype=torch.float32, device=dev)
    ref = cuda_lib.paged_e4m3(q, kc, vc, ks, vs, bt, p.ctx_len, p.scale)
    torch.cuda.synchronize()
    lib = binding.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    num_pages, page, Hkv, D = kc.shape
    # Same split partition as the workspace entry point while the device has
    # at most 160 SMs (the static array's split limit): bitwise equal output.
    same_splits = torch.cuda.get_device_properties(dev).multi_processor_count <= 160
    oracle_ref = None
    if R in (1, 8):
        import oracle
        oracle_ref = oracle.paged_e4m3(p.q, p.kcache, p.vcache, p.kscale, p.vscale,
                                       p.block_table, p.ctx_len, p.scale)
    for _ in range(2):
        out = torch.full_like(q, float("nan"))
        st = lib.gqa_attn_paged_e4m3_noalloc(
            ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(kc.data_ptr()),
            ctypes.c_void_p(vc.data_ptr()), ctypes.c_void_p(ks.data_ptr()),
            ctypes.c_void_p(vs.data_ptr()), ctypes.c_void_p(bt.data_ptr()), num_pages, page,
            p.ctx_len, R, 6, Hkv, D, p.scale, ctypes.c_void_p(out.data_ptr()), stream)
        assert st == binding.GQA_OK, binding.status_string(st)
        torch.cuda.synchronize()
        assert binding.device_error() == 0
        _close(out, ref)
        if same_splits:
            assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
        if oracle_ref is not None:
            _close_to_oracle(out, oracle_ref)


def test_noalloc_rejects_more_than_eight_rows(cuda_lib):
    lib = binding.load()
    fake = ctypes.c_void_p(0x10000)
    st = lib.gqa_attn_paged_e4m3_noalloc(fake, fake, fake, fake, fake, fake, 64, 16, 100, 9, 6, 1,
                                         256, 0.0625, fake, None)
    assert st == binding.GQA_ERR_UNSUPPORTED
