"""Oracle for BSR (paged) KV-cache attention — TEST INFRASTRUCTURE ONLY.

A plain, slow fp64 CPU statement of what the GPU path computes, written from
"FlashInfer: Block-Sparse KV 캐시로 어텐션 병목을 해소하다 (MLSys 2025 Best
Paper)" (visionhong.com), sections "FlashInfer는 KV 캐시를 어떻게 통합하는가?:
Block-Sparse 포맷" (BSR blocks, paged/contiguous as instances, inactive-block
skipping, shared-prefix composition), "어텐션 연산에서 진짜 병목은 어디인가?"
(decode vs prefill) and "JIT 컴파일은 어텐션을 어떻게 빠르게 만드는가?" (RoPE
fused into attention).  The arithmetic lives in ``bsr_oracle.c`` (plain C,
fp64, OpenMP over output rows); this module compiles it with gcc on first use
and marshals numpy arrays through ctypes.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  It shares no code with the CUDA library and
never imports it.

Pins (tests/test_oracle.py): torch CPU fp64 dense attention on tiny inputs,
closed forms (L = 1, q = 0, equal keys), page-size and page-permutation
invariance, block dropping == masking, split + merge == unsplit,
cascade == flat, causal rows == shorter decode, RoPE == complex rotation.
"""
from __future__ import annotations

import contextlib
import ctypes
import hashlib
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bsr_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_lock = threading.Lock()
_lib = None

_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_f64p = ctypes.POINTER(ctypes.c_double)


def _so_path() -> str:
    with open(_SRC, "rb") as f:
        tag = hashlib.sha1(f.read()).hexdigest()[:12]
    return os.path.join(_BUILD, f"liboracle_{tag}.so")


def build() -> str:
    """Compile the C oracle (gcc, -O2, OpenMP) if it is missing; return the .so path."""
    so = _so_path()
    if os.path.exists(so):
        return so
    os.makedirs(_BUILD, exist_ok=True)
    tmp = f"{so}.{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, so)
    return so


def _configure(lib):
    lib.oracle_attention.restype = ctypes.c_int
    lib.oracle_attention.argtypes = [
        _u16p, _u16p, _u16p, _i32p, _i32p, _i32p, _i32p,
        ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
        ctypes.c_int64, ctypes.c_double, ctypes.c_double, ctypes.c_int32, ctypes.c_int32,
        _i32p, ctypes.c_int32, _i64p, _i32p, ctypes.c_int64, _f64p, _f64p, ctypes.c_int32]
    lib.oracle_attention_kv8.restype = ctypes.c_int
    lib.oracle_attention_kv8.argtypes = [
        _u16p, _u8p, _u8p, ctypes.c_double, ctypes.c_double, _i32p, _i32p, _i32p, _i32p,
        ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
        ctypes.c_int64, ctypes.c_double, ctypes.c_double, ctypes.c_int32, ctypes.c_int32,
        _i32p, ctypes.c_int32, _i64p, _i32p, ctypes.c_int64, _f64p, _f64p, ctypes.c_int32]
    lib.oracle_e4m3.restype = ctypes.c_double
    lib.oracle_e4m3.argtypes = [ctypes.c_uint8]
    lib.oracle_merge_states.restype = None
    lib.oracle_merge_states.argtypes = [_f64p, _f64p, _f64p, _f64p, ctypes.c_int64,
                                        ctypes.c_int32, _f64p, _f64p]
    lib.oracle_append_kv.restype = ctypes.c_int
    lib.oracle_append_kv.argtypes = [_u16p, _u16p, _i32p, _i32p, _i32p, _i32p,
                                     ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                     ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, _u16p,
                                     _u16p]
    lib.oracle_kv_len.restype = ctypes.c_int
    lib.oracle_kv_len.argtypes = [_i32p, _i32p, ctypes.c_int32, ctypes.c_int32, _i64p]
    lib.oracle_rope.restype = None
    lib.oracle_rope.argtypes = [_f64p, _f64p, ctypes.c_int32, ctypes.c_double,
                                ctypes.c_double]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _configure(ctypes.CDLL(build()))
    return _lib


@contextlib.contextmanager
def _library(path: str):
    """Route every oracle call through another build of the C source (used by the
    tests that plant mistakes in a copy of the oracle and expect a pin to catch them)."""
    global _lib
    with _lock:
        prev = _lib
        _lib = _configure(ctypes.CDLL(path))
    try:
        yield
    finally:
        with _lock:
            _lib = prev


def _bits(x) -> np.ndarray:
    """bf16 data as a contiguous uint16 numpy array of its bit patterns."""
    if hasattr(x, "view") and hasattr(x, "dtype") and str(x.dtype) == "torch.bfloat16":
        import torch
        x = x.detach().contiguous().view(torch.int16).numpy()
    a = np.ascontiguousarray(x)
    if a.dtype == np.int16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError(f"expected bf16 bits, got {a.dtype}")
    return a


def _i32(x) -> np.ndarray:
    if hasattr(x, "numpy"):
        x = x.numpy()
    return np.ascontiguousarray(x, dtype=np.int32)


def _ptr(a: np.ndarray, t):
    return a.ctypes.data_as(t)


def _layout_code(kv_layout: str) -> int:
    if kv_layout not in ("HND", "NHD"):
        raise ValueError("kv_layout must be 'HND' or 'NHD'")
    return 1 if kv_layout == "NHD" else 0


def default_threads() -> int:
    return len(os.sched_getaffinity(0))


def _codes(x) -> np.ndarray:
    """FP8 (E4M3) data as a contiguous uint8 numpy array of its codes."""
    if hasattr(x, "numpy"):
        x = x.detach().contiguous()
        if str(x.dtype) != "torch.uint8":
            import torch
            x = x.view(torch.uint8)
        x = x.numpy()
    a = np.ascontiguousarray(x)
    if a.dtype != np.uint8:
        raise TypeError(f"expected E4M3 codes as uint8, got {a.dtype}")
    return a


def e4m3(codes) -> np.ndarray:
    """Values (fp64) of OCP FP8 E4M3 codes (NaN for S.1111.111)."""
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8).ravel()
    return np.array([lib.oracle_e4m3(int(v)) for v in c], dtype=np.float64).reshape(np.shape(codes))


def attention(q, k_pages, v_pages, indptr, indices, last_page_len, qo_indptr, *,
              num_qo_heads: int, num_kv_heads: int, head_dim: int, page_size: int,
              sm_scale: float, rope_theta: float = 0.0, causal: bool = False,
              window_left: int = 0, page_pos=None, kv_layout: str = "HND", rows=None,
              heads=None, threads: int | None = None):
    """Exact (fp64) attention over a paged KV cache.

    ``q`` is bf16 [sum_qo, Hq, D]; ``k_pages``/``v_pages`` are bf16
    [num_pages, Hk, P, D] (torch bf16 tensors or uint16 bit arrays).  With
    ``rows``/``heads`` given, only those (query row, qo head) pairs are
    computed and returned in that order; otherwise all of them.
    Returns ``(out [n, D] float64, lse [n] float64)``; for the full case the
    arrays are reshaped to ``[sum_qo, Hq, D]`` and ``[sum_qo, Hq]``.
    ``window_left`` > 0 restricts a query at position p to keys p - window_left + 1 .. p
    (sliding window; with causal the upper bound is p, else the request's end).
    ``page_pos`` (int32 [len(indices)]): logical position of each page's first token,
    for RoPE over caches whose dropped blocks leave gaps (default: the cached order).
    ``kv_layout``: "HND" pages [num_pages, Hk, P, D] or "NHD" pages [num_pages, P, Hk, D].
    """
    return _attention(None, q, k_pages, v_pages, indptr, indices, last_page_len, qo_indptr,
                      num_qo_heads, num_kv_heads, head_dim, page_size, sm_scale, rope_theta,
                      causal, window_left, page_pos, kv_layout, rows, heads, threads)


def attention_kv8(q, k_pages, v_pages, k_scale: float, v_scale: float, indptr, indices,
                  last_page_len, qo_indptr, *, num_qo_heads: int, num_kv_heads: int,
                  head_dim: int, page_size: int, sm_scale: float, rope_theta: float = 0.0,
                  causal: bool = False, window_left: int = 0, page_pos=None,
                  kv_layout: str = "HND", rows=None, heads=None, threads: int | None = None):
    """:func:`attention` over an FP8 KV cache: ``k_pages``/``v_pages`` hold E4M3
    codes (uint8, same layout) and the keys / values are ``k_scale * code`` and
    ``v_scale * code``."""
    return _attention((float(k_scale), float(v_scale)), q, k_pages, v_pages, indptr, indices,
                      last_page_len, qo_indptr, num_qo_heads, num_kv_heads, head_dim,
                      page_size, sm_scale, rope_theta, causal, window_left, page_pos, kv_layout,
                      rows, heads, threads)


def _attention(kv8, q, k_pages, v_pages, indptr, indices, last_page_len, qo_indptr,
               num_qo_heads, num_kv_heads, head_dim, page_size, sm_scale, rope_theta, causal,
               window_left, page_pos, kv_layout, rows, heads, threads):
    lib = _load()
    qb = _bits(q)
    if kv8 is None:
        kb, vb = _bits(k_pages), _bits(v_pages)
    else:
        kb, vb = _codes(k_pages), _codes(v_pages)
    ip, ix, lp, qi = _i32(indptr), _i32(indices), _i32(last_page_len), _i32(qo_indptr)
    batch = len(ip) - 1
    num_pages = kb.size // (num_kv_heads * page_size * head_dim)
    sum_qo = int(qi[-1])
    if rows is not None:
        sr = np.ascontiguousarray(rows, dtype=np.int64)
        sh = np.ascontiguousarray(heads, dtype=np.int32)
        n = len(sr)
        srp, shp = _ptr(sr, _i64p), _ptr(sh, _i32p)
    else:
        n = sum_qo * num_qo_heads
        srp, shp = None, None
    out = np.zeros((n, head_dim), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    if len(ix) == 0:
        ix = np.zeros((1,), dtype=np.int32)
    pp = None
    if page_pos is not None:
        pp = _i32(page_pos)
        if len(pp) != len(ix) and not (len(pp) == 0 and int(ip[-1]) == 0):
            raise ValueError("page_pos needs one entry per page-table entry")
    table = (_ptr(ip, _i32p), _ptr(ix, _i32p), _ptr(lp, _i32p) if len(lp) else None,
             _ptr(qi, _i32p), batch, num_qo_heads, num_kv_heads, head_dim, page_size, num_pages,
             float(sm_scale), float(rope_theta), int(bool(causal)), int(window_left),
             _ptr(pp, _i32p) if pp is not None else None, _layout_code(kv_layout), srp, shp, n,
             _ptr(out, _f64p), _ptr(lse, _f64p), int(threads or default_threads()))
    if kv8 is None:
        rc = lib.oracle_attention(_ptr(qb, _u16p), _ptr(kb, _u16p), _ptr(vb, _u16p), *table)
    else:
        rc = lib.oracle_attention_kv8(_ptr(qb, _u16p), _ptr(kb, _u8p), _ptr(vb, _u8p),
                                      kv8[0], kv8[1], *table)
    if rc != 0:
        raise ValueError("oracle_attention: malformed input")
    if rows is None:
        return out.reshape(sum_qo, num_qo_heads, head_dim), lse.reshape(sum_qo, num_qo_heads)
    return out, lse


def merge_states(o_a, lse_a, o_b, lse_b):
    """LSE merge of two states over disjoint key sets (fp64)."""
    lib = _load()
    o_a = np.ascontiguousarray(o_a, dtype=np.float64)
    o_b = np.ascontiguousarray(o_b, dtype=np.float64)
    la = np.ascontiguousarray(lse_a, dtype=np.float64)
    lb = np.ascontiguousarray(lse_b, dtype=np.float64)
    D = o_a.shape[-1]
    n = la.size
    o = np.zeros_like(o_a)
    l = np.zeros_like(la)
    lib.oracle_merge_states(_ptr(o_a, _f64p), _ptr(la, _f64p), _ptr(o_b, _f64p),
                            _ptr(lb, _f64p), n, D, _ptr(o, _f64p), _ptr(l, _f64p))
    return o, l


def append_kv(k_new, v_new, append_indptr, indptr, indices, last_page_len, k_pages, v_pages, *,
              num_kv_heads: int, head_dim: int, page_size: int, kv_layout: str = "HND"):
    """Return copies of the page pools with the new tokens written in (bit exact)."""
    lib = _load()
    kn, vn = _bits(k_new), _bits(v_new)
    kp, vp = _bits(k_pages).copy(), _bits(v_pages).copy()
    ai, ip, ix, lp = _i32(append_indptr), _i32(indptr), _i32(indices), _i32(last_page_len)
    batch = len(ip) - 1
    num_pages = kp.size // (num_kv_heads * page_size * head_dim)
    rc = lib.oracle_append_kv(_ptr(kn, _u16p), _ptr(vn, _u16p), _ptr(ai, _i32p),
                              _ptr(ip, _i32p), _ptr(ix, _i32p), _ptr(lp, _i32p), batch,
                              num_kv_heads, head_dim, page_size, num_pages,
                              _layout_code(kv_layout), _ptr(kp, _u16p), _ptr(vp, _u16p))
    if rc != 0:
        raise ValueError("oracle_append_kv: malformed input")
    return kp, vp


def kv_len(indptr, last_page_len, page_size: int) -> np.ndarray:
    """Attended KV length per request from the page table."""
    lib = _load()
    ip, lp = _i32(indptr), _i32(last_page_len)
    batch = len(ip) - 1
    out = np.zeros((batch,), dtype=np.int64)
    if lib.oracle_kv_len(_ptr(ip, _i32p), _ptr(lp, _i32p) if batch else None, batch,
                         page_size, _ptr(out, _i64p)) != 0:
        raise ValueError("oracle_kv_len: malformed page table")
    return out


def rope(x, pos: float, theta: float) -> np.ndarray:
    """Rotate-half RoPE of one D-vector at position ``pos`` (fp64)."""
    lib = _load()
    xi = np.ascontiguousarray(x, dtype=np.float64)
    xo = np.zeros_like(xi)
    lib.oracle_rope(_ptr(xi, _f64p), _ptr(xo, _f64p), xi.size, float(pos), float(theta))
    return xo


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to bf16 (round to nearest even via fp32), returned as float64.

    Two roundings (fp64 -> fp32 -> bf16) can differ from a single one only in
    ties below fp32 resolution; the comparison it serves tolerates that.
    """
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    r = np.where(np.isnan(f), np.uint64(0x7FC00000), r)
    return r.astype(np.uint32).view(np.float32).astype(np.float64)
