"""FP64 CPU oracle for causal GQA attention (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s cpu_baseline /
reference leg may import this package.  The product path (the CUDA library and
its Python binding) never does, and shares no code with it.

The arithmetic lives in ``gqa_oracle.c`` (plain C, double precision, two-pass
softmax over an explicit visible-key list); this module compiles it with gcc on
first use and marshals numpy / torch CPU arrays into it.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gqa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/liboracle.so`` (plain gcc, -O2)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC,
                               "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I = ctypes.c_int
            Dd = ctypes.c_double
            lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_decode.restype = Dd
            lib.oracle_dense.argtypes = [P, P, P, I, I, I, I, I, Dd, P, I, P, I]
            lib.oracle_dense.restype = I
            lib.oracle_paged_e4m3.argtypes = [P, P, P, Dd, Dd, P, I, I, I, I, I, I, Dd, P, I,
                                              P, I]
            lib.oracle_paged_e4m3.restype = I
            lib.oracle_sparse_blocks.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, Dd, P,
                                                 I, P, I]
            lib.oracle_sparse_blocks.restype = I
            lib.oracle_sparse_blocks_e4m3.argtypes = [P, P, P, Dd, Dd, P, P, P, I, I, I, I, I,
                                                      I, I, Dd, P, I, P, I]
            lib.oracle_sparse_blocks_e4m3.restype = I
            lib.oracle_dense_probs.argtypes = [P, P, P, I, I, I, I, I, Dd, I, I, P]
            lib.oracle_dense_probs.restype = I
            _lib = lib
    return _lib


def _np(x, dtype):
    """CPU contiguous numpy view of a torch tensor or array with the given dtype."""
    if hasattr(x, "detach"):
        x = x.detach().cpu().contiguous()
        if dtype == np.uint16:
            import torch
            x = x.view(torch.int16).numpy().view(np.uint16)
        elif dtype == np.uint8:
            import torch
            x = x.view(torch.uint8).numpy()
        else:
            x = x.numpy()
    x = np.ascontiguousarray(x)
    if dtype == np.uint16 and x.dtype == np.float16:
        x = x.view(np.uint16)
    assert x.dtype == dtype, (x.dtype, dtype)
    return x


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _rows(rows, total):
    if rows is None:
        rows = np.arange(total, dtype=np.int32)
    return np.ascontiguousarray(np.asarray(rows, dtype=np.int32))


def _threads(nthreads):
    return int(nthreads) if nthreads else (os.cpu_count() or 1)


def e4m3_decode(code: int) -> float:
    """Exact value of one E4M3 byte (OCP e4m3fn reading)."""
    return float(_load().oracle_e4m3_decode(int(code) & 0xFF))


def dense(q, k, v, scale: float, rows=None, nthreads=None) -> np.ndarray:
    """Dense bottom-right causal attention.

    q [Q, Hq, D], k/v [KV, Hkv, D] fp16 (torch or numpy).  Returns float64
    [len(rows), Hq, D] for the selected query rows (all rows by default).
    """
    qa, ka, va = _np(q, np.uint16), _np(k, np.uint16), _np(v, np.uint16)
    Q, Hq, D = qa.shape
    KV, Hkv, D2 = ka.shape
    assert D == D2 and va.shape == ka.shape
    r = _rows(rows, Q)
    out = np.zeros((len(r), Hq, D), dtype=np.float64)
    rc = _load().oracle_dense(_ptr(qa), _ptr(ka), _ptr(va), Q, KV, Hq, Hkv, D, float(scale),
                              _ptr(r), len(r), _ptr(out), _threads(nthreads))
    if rc:
        raise ValueError("oracle_dense: invalid arguments")
    return out


def dense_probs(q, k, v, scale: float, row: int, head: int) -> np.ndarray:
    """Normalised attention weights of one (row, head) over its visible keys."""
    qa, ka, va = _np(q, np.uint16), _np(k, np.uint16), _np(v, np.uint16)
    Q, Hq, D = qa.shape
    KV, Hkv, _ = ka.shape
    probs = np.zeros(KV, dtype=np.float64)
    n = _load().oracle_dense_probs(_ptr(qa), _ptr(ka), _ptr(va), Q, KV, Hq, Hkv, D,
                                   float(scale), int(row), int(head), _ptr(probs))
    if n < 0:
        raise ValueError("oracle_dense_probs: invalid arguments")
    return probs[:n]


def paged_e4m3(q, kcache, vcache, kscale: float, vscale: float, block_table, ctx_len: int,
               scale: float, rows=None, nthreads=None) -> np.ndarray:
    """Paged E4M3 tail: q [R, Hq, D] fp16; caches [num_pages, page, Hkv, D] uint8."""
    qa = _np(q, np.uint16)
    kc, vc = _np(kcache, np.uint8), _np(vcache, np.uint8)
    bt = _np(block_table, np.int32)
    R, Hq, D = qa.shape
    _, page, Hkv, D2 = kc.shape
    assert D == D2 and vc.shape == kc.shape
    assert bt.shape[0] * page >= ctx_len
    assert int(bt[: (ctx_len + page - 1) // page].max(initial=0)) < kc.shape[0]
    r = _rows(rows, R)
    out = np.zeros((len(r), Hq, D), dtype=np.float64)
    rc = _load().oracle_paged_e4m3(_ptr(qa), _ptr(kc), _ptr(vc), float(kscale), float(vscale),
                                   _ptr(bt), page, int(ctx_len), R, Hq, Hkv, D, float(scale),
                                   _ptr(r), len(r), _ptr(out), _threads(nthreads))
    if rc:
        raise ValueError("oracle_paged_e4m3: invalid arguments")
    return out


def dense_e4m3(q, k, v, kscale: float, vscale: float, scale: float, rows=None,
               nthreads=None) -> np.ndarray:
    """Dense bottom-right causal attention over E4M3 keys and values: the E4M3
    storage of "[Perf] Ship the qualified SM70 long-context layout and drop its
    context fences" (What) applied to the dense prefill of "[Kernel][SM70]
    Default long-prefill GQA architecture" (Purpose).  q [Q, Hq, D] fp16, k / v
    [KV, Hkv, D] uint8 E4M3 codes with real value decode(byte) * kscale /
    vscale.  The same arithmetic as the paged tail with the whole context in
    one page (block table [0]), so row i sees keys 0 .. KV - Q + i."""
    ka, va = _np(k, np.uint8), _np(v, np.uint8)
    KV, Hkv, D = ka.shape
    table = np.zeros(1, dtype=np.int32)
    return paged_e4m3(q, ka.reshape(1, KV, Hkv, D), va.reshape(1, KV, Hkv, D), kscale, vscale,
                      table, KV, scale, rows=rows, nthreads=nthreads)


def sparse_blocks(q, kcache, vcache, block_table, sel_idx, sel_cnt, ctx_len: int,
                  scale: float, rows=None, nthreads=None) -> np.ndarray:
    """Selected-block sparse attention over an fp16 page cache."""
    qa = _np(q, np.uint16)
    kc, vc = _np(kcache, np.uint16), _np(vcache, np.uint16)
    bt = _np(block_table, np.int32)
    si, sc = _np(sel_idx, np.int32), _np(sel_cnt, np.int32)
    n_rows, Hq, D = qa.shape
    _, page, Hkv, D2 = kc.shape
    assert D == D2 and vc.shape == kc.shape
    assert si.shape[0] == n_rows and sc.shape[0] == n_rows
    assert bt.shape[0] * page >= ctx_len
    max_sel = si.shape[1]
    r = _rows(rows, n_rows)
    out = np.zeros((len(r), Hq, D), dtype=np.float64)
    rc = _load().oracle_sparse_blocks(_ptr(qa), _ptr(kc), _ptr(vc), _ptr(bt), _ptr(si),
                                      _ptr(sc), max_sel, page, int(ctx_len), n_rows, Hq, Hkv,
                                      D, float(scale), _ptr(r), len(r), _ptr(out),
                                      _threads(nthreads))
    if rc:
        raise ValueError("oracle_sparse_blocks: invalid arguments")
    return out


def sparse_blocks_e4m3(q, kcache, vcache, kscale: float, vscale: float, block_table, sel_idx,
                       sel_cnt, ctx_len: int, scale: float, rows=None, nthreads=None) -> np.ndarray:
    """Selected-block sparse attention over an E4M3 page cache (uint8 codes,
    values decode(byte) * kscale / vscale)."""
    qa = _np(q, np.uint16)
    kc, vc = _np(kcache, np.uint8), _np(vcache, np.uint8)
    bt = _np(block_table, np.int32)
    si, sc = _np(sel_idx, np.int32), _np(sel_cnt, np.int32)
    n_rows, Hq, D = qa.shape
    _, page, Hkv, D2 = kc.shape
    assert D == D2 and vc.shape == kc.shape
    assert si.shape[0] == n_rows and sc.shape[0] == n_rows
    assert bt.shape[0] * page >= ctx_len
    max_sel = si.shape[1]
    r = _rows(rows, n_rows)
    out = np.zeros((len(r), Hq, D), dtype=np.float64)
    rc = _load().oracle_sparse_blocks_e4m3(_ptr(qa), _ptr(kc), _ptr(vc), float(kscale),
                                           float(vscale), _ptr(bt), _ptr(si), _ptr(sc), max_sel,
                                           page, int(ctx_len), n_rows, Hq, Hkv, D, float(scale),
                                           _ptr(r), len(r), _ptr(out), _threads(nthreads))
    if rc:
        raise ValueError("oracle_sparse_blocks_e4m3: invalid arguments")
    return out
