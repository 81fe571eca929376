"""Python binding of libgqa_attn.so (ctypes; argument marshalling only).

Every function here forwards torch tensors' device pointers, shapes and the
current CUDA stream to the C ABI declared in ``include/gqa_attn.h``; all of the
attention runs in the library's CUDA kernels.  There is no fallback: if the
library is missing or a call fails, a ``GQAError`` is raised.

Workspace: the prefill and paged-E4M3 entry points keep split partials in a
workspace registered per device.  ``ensure_workspace`` allocates it with torch
(outside the C calls) and registers it; the wrappers call it for you.
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libgqa_attn.so")

GQA_OK = 0
GQA_ERR_INVALID_ARG = 1
GQA_ERR_UNSUPPORTED = 2
GQA_ERR_WORKSPACE = 3
GQA_ERR_CUDA = 4
KIND_PREFILL = 0
KIND_PAGED_E4M3 = 1
KIND_SPARSE = 2
KIND_PAGED_E4M3_BATCH = 3
DEVERR_WAIT_TIMEOUT = 0x1
DEVERR_BAD_BLOCK_ID = 0x2
DEVERR_BAD_PAGE_ID = 0x4
DEVERR_BAD_CTX_LEN = 0x8
DEVERR_DUP_BLOCK_ID = 0x10

# Every symbol include/gqa_attn.h declares.
EXPORTED = ("gqa_attn_prefill", "gqa_attn_prefill_e4m3", "gqa_attn_paged_e4m3", "gqa_attn_paged_e4m3_devctx",
            "gqa_attn_paged_e4m3_batch",
            "gqa_attn_paged_e4m3_noalloc",
            "gqa_attn_sparse_blocks", "gqa_attn_sparse_blocks_e4m3",
            "gqa_workspace_bytes", "gqa_set_workspace", "gqa_get_device_error",
            "gqa_check_wait_limit", "gqa_prefill_sm_pairs", "gqa_status_string")


class GQAError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


_lock = threading.Lock()
_lib = None
_ws = {}  # device index -> torch.uint8 tensor registered as workspace


def load():
    """Load libgqa_attn.so (it must have been built; see build_lib.build)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise GQAError(GQA_ERR_CUDA, f"{LIB_PATH} not built")
            lib = ctypes.CDLL(LIB_PATH)
            P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
            lib.gqa_attn_prefill.argtypes = [P, P, P, P, I, I, I, I, I, F, P]
            lib.gqa_attn_prefill.restype = I
            lib.gqa_attn_prefill_e4m3.argtypes = [P, P, P, P, P, P, I, I, I, I, I, F, P]
            lib.gqa_attn_prefill_e4m3.restype = I
            lib.gqa_attn_paged_e4m3.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, F, P, P]
            lib.gqa_attn_paged_e4m3.restype = I
            lib.gqa_attn_paged_e4m3_devctx.argtypes = [P, P, P, P, P, P, I, I, P, I, I, I, I, I,
                                                       F, P, P]
            lib.gqa_attn_paged_e4m3_devctx.restype = I
            lib.gqa_attn_paged_e4m3_batch.argtypes = [P, P, P, P, P, P, I, I, I, P, I, I, I, I, I,
                                                      I, F, P, P]
            lib.gqa_attn_paged_e4m3_batch.restype = I
            lib.gqa_attn_paged_e4m3_noalloc.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I,
                                                        F, P, P]
            lib.gqa_attn_paged_e4m3_noalloc.restype = I
            lib.gqa_attn_sparse_blocks.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, I, F,
                                                   P, P]
            lib.gqa_attn_sparse_blocks.restype = I
            lib.gqa_attn_sparse_blocks_e4m3.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I,
                                                        I, I, I, F, P, P]
            lib.gqa_attn_sparse_blocks_e4m3.restype = I
            lib.gqa_workspace_bytes.argtypes = [I, I, I, I, I]
            lib.gqa_workspace_bytes.restype = Z
            lib.gqa_set_workspace.argtypes = [I, P, Z]
            lib.gqa_set_workspace.restype = I
            lib.gqa_get_device_error.argtypes = [P]
            lib.gqa_get_device_error.restype = I
            lib.gqa_check_wait_limit.argtypes = [P]
            lib.gqa_check_wait_limit.restype = I
            lib.gqa_prefill_sm_pairs.argtypes = []
            lib.gqa_prefill_sm_pairs.restype = I
            lib.gqa_status_string.argtypes = [I]
            lib.gqa_status_string.restype = ctypes.c_char_p
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().gqa_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != GQA_OK:
        raise GQAError(status, what)


def _stream_ptr(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t: torch.Tensor):
    return ctypes.c_void_p(t.data_ptr())


def _need_cuda(*ts):
    dev = None
    for t in ts:
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise GQAError(GQA_ERR_INVALID_ARG, "tensors must be CUDA tensors")
        if not t.is_contiguous():
            raise GQAError(GQA_ERR_INVALID_ARG, "tensors must be contiguous")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise GQAError(GQA_ERR_INVALID_ARG, "tensors on different devices")
    return dev


def workspace_bytes(kind: int, query_rows: int, ctx_or_kv: int, Hq: int = 6, D: int = 256) -> int:
    return int(load().gqa_workspace_bytes(kind, query_rows, ctx_or_kv, Hq, D))


def ensure_workspace(nbytes: int, device=None) -> torch.Tensor:
    """Make sure the device's registered workspace holds at least nbytes."""
    dev = torch.device(device if device is not None else "cuda")
    idx = dev.index if dev.index is not None else torch.cuda.current_device()
    cur = _ws.get(idx)
    if cur is None or cur.numel() < nbytes:
        torch.cuda.synchronize(idx)
        buf = torch.empty(max(int(nbytes), 4096), dtype=torch.uint8, device=f"cuda:{idx}")
        _check(load().gqa_set_workspace(idx, _ptr(buf), buf.numel()), "gqa_set_workspace")
        _ws[idx] = buf
        cur = buf
    return cur


def register_workspace(buf: torch.Tensor):
    """Register a caller-provided uint8 CUDA buffer as its device's workspace."""
    _need_cuda(buf)
    idx = buf.device.index
    _check(load().gqa_set_workspace(idx, _ptr(buf), buf.numel()), "gqa_set_workspace")
    _ws[idx] = buf


def device_error(stream=None) -> int:
    """Synchronise the stream and read-and-clear the device error word."""
    v = load().gqa_get_device_error(_stream_ptr(stream))
    if v < 0:
        raise GQAError(GQA_ERR_CUDA, "gqa_get_device_error")
    return v


def check_wait_limit(stream=None) -> None:
    """Queue the bounded-wait diagnostic (gqa_check_wait_limit): a wait on an
    mbarrier nothing arrives on, which gives up after its limit and sets
    DEVERR_WAIT_TIMEOUT; read it with device_error()."""
    st = load().gqa_check_wait_limit(_stream_ptr(stream))
    if st != GQA_OK:
        raise GQAError(st, "gqa_check_wait_limit")


def prefill_sm_pairs() -> int:
    """SM pairs the dense prefill kernel runs on (co-resident two-CTA clusters)."""
    v = load().gqa_prefill_sm_pairs()
    if v < 0:
        raise GQAError(GQA_ERR_CUDA, "gqa_prefill_sm_pairs")
    return v


def prefill(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: float = 1.0 / 16,
            out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Dense causal GQA prefill: q [Q,Hq,D], k/v [KV,Hkv,D] fp16 -> out [Q,Hq,D]."""
    dev = _need_cuda(q, k, v)
    Q, Hq, D = q.shape
    KV, Hkv, _ = k.shape
    if out is None:
        out = torch.empty_like(q)
    _need_cuda(out)
    with torch.cuda.device(dev):
        ensure_workspace(workspace_bytes(KIND_PREFILL, Q, KV, Hq, D), dev)
        st = load().gqa_attn_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(out), Q, KV, Hq, Hkv, D,
                                     float(scale), _stream_ptr(stream))
    _check(st, "gqa_attn_prefill")
    return out


def prefill_e4m3(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, kscale: torch.Tensor,
                 vscale: torch.Tensor, scale: float = 1.0 / 16, out: torch.Tensor | None = None,
                 stream=None) -> torch.Tensor:
    """Dense causal GQA prefill over an E4M3 K/V cache: q [Q,Hq,D] fp16, k/v
    [KV,Hkv,D] uint8 codes, kscale/vscale one-element fp32 CUDA tensors."""
    dev = _need_cuda(q, k, v, kscale, vscale)
    Q, Hq, D = q.shape
    KV, Hkv, _ = k.shape
    if out is None:
        out = torch.empty_like(q)
    _need_cuda(out)
    with torch.cuda.device(dev):
        ensure_workspace(workspace_bytes(KIND_PREFILL, Q, KV, Hq, D), dev)
        st = load().gqa_attn_prefill_e4m3(_ptr(q), _ptr(k), _ptr(v), _ptr(kscale), _ptr(vscale),
                                          _ptr(out), Q, KV, Hq, Hkv, D, float(scale),
                                          _stream_ptr(stream))
    _check(st, "gqa_attn_prefill_e4m3")
    return out


def paged_e4m3(q: torch.Tensor, kcache: torch.Tensor, vcache: torch.Tensor,
               kscale: torch.Tensor, vscale: torch.Tensor, block_table: torch.Tensor,
               ctx_len: int, scale: float = 1.0 / 16, out: torch.Tensor | None = None,
               stream=None) -> torch.Tensor:
    """Paged E4M3 verifier tail: q [R,Hq,D] fp16, caches [pages,page,Hkv,D] uint8,
    kscale/vscale one-element fp32 CUDA tensors, block_table int32."""
    dev = _need_cuda(q, kcache, vcache, kscale, vscale, block_table)
    R, Hq, D = q.shape
    num_pages, page, Hkv, _ = kcache.shape
    if out is None:
        out = torch.empty_like(q)
    _need_cuda(out)
    with torch.cuda.device(dev):
        ensure_workspace(workspace_bytes(KIND_PAGED_E4M3, R, ctx_len, Hq, D), dev)
        st = load().gqa_attn_paged_e4m3(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(kscale),
                                        _ptr(vscale), _ptr(block_table), num_pages, page,
                                        int(ctx_len), R, Hq, Hkv, D, float(scale), _ptr(out),
                                        _stream_ptr(stream))
    _check(st, "gqa_attn_paged_e4m3")
    return out


def paged_e4m3_devctx(q: torch.Tensor, kcache: torch.Tensor, vcache: torch.Tensor,
                      kscale: torch.Tensor, vscale: torch.Tensor, block_table: torch.Tensor,
                      ctx_len_dev: torch.Tensor, max_ctx_len: int, scale: float = 1.0 / 16,
                      out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Paged E4M3 tail with the context length read on the device when the
    kernels run: ctx_len_dev is a one-element int32 CUDA tensor, max_ctx_len
    the host bound that sizes the grid and the workspace."""
    dev = _need_cuda(q, kcache, vcache, kscale, vscale, block_table, ctx_len_dev)
    if ctx_len_dev.dtype != torch.int32 or ctx_len_dev.numel() < 1:
        raise GQAError(GQA_ERR_INVALID_ARG, "ctx_len_dev must be a CUDA int32 tensor")
    R, Hq, D = q.shape
    num_pages, page, Hkv, _ = kcache.shape
    if out is None:
        out = torch.empty_like(q)
    _need_cuda(out)
    with torch.cuda.device(dev):
        ensure_workspace(workspace_bytes(KIND_PAGED_E4M3, R, max_ctx_len, Hq, D), dev)
        st = load().gqa_attn_paged_e4m3_devctx(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(kscale),
                                               _ptr(vscale), _ptr(block_table), num_pages, page,
                                               _ptr(ctx_len_dev), int(max_ctx_len), R, Hq, Hkv, D,
                                               float(scale), _ptr(out), _stream_ptr(stream))
    _check(st, "gqa_attn_paged_e4m3_devctx")
    return out


def paged_e4m3_batch(q: torch.Tensor, kcache: torch.Tensor, vcache: torch.Tensor,
                     kscale: torch.Tensor, vscale: torch.Tensor, block_tables: torch.Tensor,
                     ctx_lens_dev: torch.Tensor, max_ctx_len: int, scale: float = 1.0 / 16,
                     out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Batched variable-length E4M3 tails: q [B,R,Hq,D] fp16, one shared page
    cache, block_tables [B, stride] int32, ctx_lens_dev [B] CUDA int32 read when
    the kernels run, max_ctx_len the host bound."""
    dev = _need_cuda(q, kcache, vcache, kscale, vscale, block_tables, ctx_lens_dev)
    if ctx_lens_dev.dtype != torch.int32 or block_tables.dtype != torch.int32:
        raise GQAError(GQA_ERR_INVALID_ARG, "ctx_lens_dev and block_tables must be int32")
    B, R, Hq, D = q.shape
    if ctx_lens_dev.numel() != B or block_tables.shape[0] != B or not block_tables.is_contiguous():
        raise GQAError(GQA_ERR_INVALID_ARG, "one context length and table row per sequence")
    num_pages, page, Hkv, _ = kcache.shape
    if out is None:
        out = torch.empty_like(q)
    _need_cuda(out)
    with torch.cuda.device(dev):
        ensure_workspace(workspace_bytes(KIND_PAGED_E4M3_BATCH, R, B, Hq, D), dev)
        st = load().gqa_attn_paged_e4m3_batch(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(kscale),
                                              _ptr(vscale), _ptr(block_tables),
                                              block_tables.shape[1], num_pages, page,
                                              _ptr(ctx_lens_dev), int(max_ctx_len), B, R, Hq, Hkv,
                                              D, float(scale), _ptr(out), _stream_ptr(stream))
    _check(st, "gqa_attn_paged_e4m3_batch")
    return out


def sparse_blocks(q: torch.Tensor, kcache: torch.Tensor, vcache: torch.Tensor,
                  block_table: torch.Tensor, sel_idx: torch.Tensor, sel_cnt: torch.Tensor,
                  ctx_len: int, scale: float = 1.0 / 16, out: torch.Tensor | None = None,
                  stream=None) -> torch.Tensor:
    """Selected-block sparse paged prefill over an fp16 page cache."""
    dev = _need_cuda(q, kcache, vcache, block_table, sel_idx, sel_cnt)
    rows, Hq, D = q.shape
    num_pages, page, Hkv, _ = kcache.shape
    max_sel = sel_idx.shape[1]
    if out is None:
        out = torch.empty_like(q)
    _need_cuda(out)
    with torch.cuda.device(dev):
        st = load().gqa_attn_sparse_blocks(_ptr(q), _ptr(kcache), _ptr(vcache),
                                           _ptr(block_table), _ptr(sel_idx), _ptr(sel_cnt),
                                           max_sel, num_pages, page, int(ctx_len), rows, Hq,
                                           Hkv, D, float(scale), _ptr(out), _stream_ptr(stream))
    _check(st, "gqa_attn_sparse_blocks")
    return out


def sparse_blocks_e4m3(q: torch.Tensor, kcache: torch.Tensor, vcache: torch.Tensor,
                       kscale: torch.Tensor, vscale: torch.Tensor, block_table: torch.Tensor,
                       sel_idx: torch.Tensor, sel_cnt: torch.Tensor, ctx_len: int,
                       scale: float = 1.0 / 16, out: torch.Tensor | None = None,
                       stream=None) -> torch.Tensor:
    """Selected-block sparse paged prefill over an E4M3 page cache: caches
    [pages,page,Hkv,D] uint8 codes, kscale/vscale one-element fp32 CUDA tensors."""
    dev = _need_cuda(q, kcache, vcache, kscale, vscale, block_table, sel_idx, sel_cnt)
    rows, Hq, D = q.shape
    num_pages, page, Hkv, _ = kcache.shape
    max_sel = sel_idx.shape[1]
    if out is None:
        out = torch.empty_like(q)
    _need_cuda(out)
    with torch.cuda.device(dev):
        st = load().gqa_attn_sparse_blocks_e4m3(_ptr(q), _ptr(kcache), _ptr(vcache),
                                                _ptr(kscale), _ptr(vscale), _ptr(block_table),
                                                _ptr(sel_idx), _ptr(sel_cnt), max_sel, num_pages,
                                                page, int(ctx_len), rows, Hq, Hkv, D,
                                                float(scale), _ptr(out), _stream_ptr(stream))
    _check(st, "gqa_attn_sparse_blocks_e4m3")
    return out
