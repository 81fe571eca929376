"""Host-side checks of the C ABI (no GPU needed).

The library must build, load and export every function include/gqa_attn.h
declares; argument validation must reject bad calls before anything reaches
the GPU.
"""

import ctypes
import os
import re

import pytest

from long_context_causal_gqa_gb300 import binding, build_lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gqa_attn.h")


@pytest.fixture(scope="module")
def lib():
    build_lib.build()
    return binding.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gqa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    assert set(names) == set(binding.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert binding.status_string(0) == "GQA_OK"
    assert binding.status_string(2) == "GQA_ERR_UNSUPPORTED"
    assert binding.status_string(99) == "GQA_UNKNOWN_STATUS"


P = ctypes.c_void_p
FAKE = P(0x10000)        # 16-byte aligned non-null stand-in; never dereferenced
FAKE_ODD = P(0x10008)    # 8-byte aligned only


def _prefill(lib, q=FAKE, Q=8, KV=16, Hq=6, Hkv=1, D=256, scale=0.0625):
    return lib.gqa_attn_prefill(q, FAKE, FAKE, FAKE, Q, KV, Hq, Hkv, D, scale, None)


def test_prefill_rejects_bad_arguments(lib):
    assert _prefill(lib, q=P(0)) == binding.GQA_ERR_INVALID_ARG
    assert _prefill(lib, q=FAKE_ODD) == binding.GQA_ERR_INVALID_ARG
    assert _prefill(lib, Q=17, KV=16) == binding.GQA_ERR_INVALID_ARG
    assert _prefill(lib, Q=0) == binding.GQA_ERR_INVALID_ARG
    assert _prefill(lib, scale=0.0) == binding.GQA_ERR_INVALID_ARG
    assert _prefill(lib, scale=float("nan")) == binding.GQA_ERR_INVALID_ARG
    assert _prefill(lib, D=64) == binding.GQA_ERR_UNSUPPORTED    # 128 and 256 are accepted
    assert _prefill(lib, D=192) == binding.GQA_ERR_UNSUPPORTED
    # Any grouping with Hkv | Hq (Hq <= 64) is accepted; these are not.
    assert _prefill(lib, Hq=7, Hkv=2) == binding.GQA_ERR_UNSUPPORTED
    assert _prefill(lib, Hq=6, Hkv=4) == binding.GQA_ERR_UNSUPPORTED
    assert _prefill(lib, Hq=65, Hkv=1) == binding.GQA_ERR_UNSUPPORTED
    assert _prefill(lib, Hkv=0) == binding.GQA_ERR_UNSUPPORTED
    assert _prefill(lib, Hq=0) == binding.GQA_ERR_UNSUPPORTED


def _paged(lib, R=8, ctx=100, pages=8, page=16, D=256, kscale=FAKE, scale=0.0625, Hq=6, Hkv=1):
    return lib.gqa_attn_paged_e4m3(FAKE, FAKE, FAKE, kscale, FAKE, FAKE, pages, page, ctx, R,
                                   Hq, Hkv, D, scale, FAKE, None)


def test_paged_rejects_bad_arguments(lib):
    assert _paged(lib, kscale=P(0)) == binding.GQA_ERR_INVALID_ARG
    assert _paged(lib, R=0) == binding.GQA_ERR_INVALID_ARG
    assert _paged(lib, R=9) == binding.GQA_ERR_UNSUPPORTED
    assert _paged(lib, D=64) == binding.GQA_ERR_UNSUPPORTED      # 128 and 256 are accepted
    assert _paged(lib, D=192) == binding.GQA_ERR_UNSUPPORTED
    assert _paged(lib, page=12) == binding.GQA_ERR_UNSUPPORTED   # not a power of two
    assert _paged(lib, page=512) == binding.GQA_ERR_UNSUPPORTED
    assert _paged(lib, page=4) == binding.GQA_ERR_UNSUPPORTED
    # One launch packs R x Hq / Hkv rows, at most 48; Hkv must divide Hq.
    assert _paged(lib, R=7, Hq=8, Hkv=1) == binding.GQA_ERR_UNSUPPORTED
    assert _paged(lib, R=17, Hq=6, Hkv=2) == binding.GQA_ERR_UNSUPPORTED
    assert _paged(lib, R=2, Hq=6, Hkv=4) == binding.GQA_ERR_UNSUPPORTED
    assert _paged(lib, R=2, Hq=6, Hkv=0) == binding.GQA_ERR_UNSUPPORTED
    assert _paged(lib, ctx=200, pages=8) == binding.GQA_ERR_INVALID_ARG  # 200 > 8 * 16
    assert _paged(lib, R=8, ctx=5) == binding.GQA_ERR_INVALID_ARG
    assert _paged(lib, scale=-1.0) == binding.GQA_ERR_INVALID_ARG


def _paged_dev(lib, R=2, max_ctx=100, pages=8, ctxp=FAKE, page=16, scale=0.0625):
    return lib.gqa_attn_paged_e4m3_devctx(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, pages, page, ctxp,
                                          max_ctx, R, 6, 1, 256, scale, FAKE, None)


def test_paged_devctx_rejects_bad_arguments(lib):
    assert _paged_dev(lib, ctxp=P(0)) == binding.GQA_ERR_INVALID_ARG
    assert _paged_dev(lib, ctxp=P(0x10002)) == binding.GQA_ERR_INVALID_ARG   # not 4-byte aligned
    assert _paged_dev(lib, R=3, max_ctx=2) == binding.GQA_ERR_INVALID_ARG
    assert _paged_dev(lib, max_ctx=200, pages=8) == binding.GQA_ERR_INVALID_ARG
    assert _paged_dev(lib, R=9, max_ctx=100) == binding.GQA_ERR_UNSUPPORTED
    assert _paged_dev(lib, page=24) == binding.GQA_ERR_UNSUPPORTED
    assert _paged_dev(lib, scale=0.0) == binding.GQA_ERR_INVALID_ARG


def _sparse(lib, rows=4, ctx=64, pages=4, max_sel=4, sel=FAKE, D=256, Hq=6, Hkv=1):
    return lib.gqa_attn_sparse_blocks(FAKE, FAKE, FAKE, FAKE, sel, FAKE, max_sel, pages, 16,
                                      ctx, rows, Hq, Hkv, D, 0.0625, FAKE, None)


def test_sparse_rejects_bad_arguments(lib):
    assert _sparse(lib, sel=P(0)) == binding.GQA_ERR_INVALID_ARG
    assert _sparse(lib, sel=P(0x10002)) == binding.GQA_ERR_INVALID_ARG
    assert _sparse(lib, max_sel=0) == binding.GQA_ERR_INVALID_ARG
    assert _sparse(lib, rows=65, ctx=64) == binding.GQA_ERR_INVALID_ARG
    assert _sparse(lib, ctx=65, pages=4) == binding.GQA_ERR_INVALID_ARG
    assert _sparse(lib, D=64) == binding.GQA_ERR_UNSUPPORTED     # 128 and 256 are accepted
    assert _sparse(lib, D=512) == binding.GQA_ERR_UNSUPPORTED
    # At most 16 query heads per KV head; Hkv must divide Hq.
    assert _sparse(lib, Hq=32, Hkv=1) == binding.GQA_ERR_UNSUPPORTED
    assert _sparse(lib, Hq=6, Hkv=4) == binding.GQA_ERR_UNSUPPORTED


def _sparse8(lib, ks=FAKE, D=256, Hq=6, Hkv=1):
    return lib.gqa_attn_sparse_blocks_e4m3(FAKE, FAKE, FAKE, ks, FAKE, FAKE, FAKE, FAKE, 4, 4,
                                           16, 64, 4, Hq, Hkv, D, 0.0625, FAKE, None)


def test_sparse_e4m3_rejects_bad_arguments(lib):
    assert _sparse8(lib, ks=P(0)) == binding.GQA_ERR_INVALID_ARG
    assert _sparse8(lib, ks=P(0x10002)) == binding.GQA_ERR_INVALID_ARG
    assert _sparse8(lib, D=64) == binding.GQA_ERR_UNSUPPORTED      # 128 and 256 are accepted
    assert _sparse8(lib, Hq=32, Hkv=1) == binding.GQA_ERR_UNSUPPORTED


def test_workspace_registration_validates(lib):
    assert lib.gqa_set_workspace(-1, None, 0) == binding.GQA_ERR_INVALID_ARG
    assert lib.gqa_set_workspace(0, P(0x10010), 1 << 20) == binding.GQA_ERR_INVALID_ARG
    assert lib.gqa_set_workspace(0, P(0x10000), 16) == binding.GQA_ERR_INVALID_ARG
    assert lib.gqa_workspace_bytes(0, 8, 16, 6, 128) == 0
    assert lib.gqa_workspace_bytes(1, 49, 100, 6, 256) == 0


def test_oracle_is_not_imported_by_the_product_path():
    pkg = os.path.join(ROOT, "long_context_causal_gqa_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".c", ".cc", ".cpp")):
                text = open(os.path.join(dirpath, f), errors="ignore").read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "gqa_oracle" not in text and "liboracle" not in text, f


def _prefill8(lib, Q=8, KV=16, D=256, Hq=6, Hkv=1, ks=FAKE, scale=0.0625):
    return lib.gqa_attn_prefill_e4m3(FAKE, FAKE, FAKE, ks, FAKE, FAKE, Q, KV, Hq, Hkv, D, scale,
                                     None)


def test_prefill_e4m3_rejects_bad_arguments(lib):
    assert _prefill8(lib, ks=P(0)) == binding.GQA_ERR_INVALID_ARG
    assert _prefill8(lib, ks=P(0x10002)) == binding.GQA_ERR_INVALID_ARG   # not 4-byte aligned
    assert _prefill8(lib, Q=17, KV=16) == binding.GQA_ERR_INVALID_ARG
    assert _prefill8(lib, scale=0.0) == binding.GQA_ERR_INVALID_ARG
    assert _prefill8(lib, D=64) == binding.GQA_ERR_UNSUPPORTED     # 128 and 256 are accepted
    assert _prefill8(lib, Hq=6, Hkv=4) == binding.GQA_ERR_UNSUPPORTED
