"""Python binding of ``libbsrattn.so``: BSR (paged) KV-cache attention on GB300.

Argument marshalling only.  Each function carries the name of the C entry
point it calls (see ``include/bsr_attn.h`` for layouts, ownership and error
behaviour); every step of the computation runs in the library's CUDA
kernels.  PyTorch supplies device memory and streams.  There is no fallback:
if the library is not built, loading it raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import _build

__all__ = [
    "BsrError", "load", "bsr_attn_plan", "bsr_attn_plan_host", "bsr_attn_run",
    "bsr_attn_run_kv8", "bsr_attn_run_host", "bsr_merge_states", "bsr_append_kv", "bsr_schedule_destroy", "bsr_schedule_get_info",
    "bsr_last_device_error", "bsr_status_string", "bsr_attn_decode_noalloc", "Schedule",
    "bsr_attn_decode_noalloc_kv8", "bsr_attn_decode_noalloc_ex",
    "bsr_schedule_set_stage_timing", "bsr_schedule_stage_times", "STAGES", "EXPORTED_SYMBOLS",
    "bsr_selftest_bounded_wait", "bsr_schedule_create",
]

BSR_OK = 0
BSR_DTYPE_BF16 = 0
BSR_DTYPE_F32 = 1

EXPORTED_SYMBOLS = (
    "bsr_attn_plan", "bsr_attn_plan_host", "bsr_attn_run", "bsr_attn_run_kv8",
    "bsr_attn_run_host", "bsr_merge_states",
    "bsr_append_kv", "bsr_schedule_destroy", "bsr_schedule_get_info", "bsr_last_device_error",
    "bsr_status_string", "bsr_attn_decode_noalloc", "bsr_attn_decode_noalloc_kv8",
    "bsr_attn_decode_noalloc_ex",
    "bsr_schedule_set_stage_timing",
    "bsr_schedule_stage_times", "bsr_selftest_bounded_wait", "bsr_schedule_create",
)

_i32p = ctypes.POINTER(ctypes.c_int32)
_vp = ctypes.c_void_p
_lib = None


class BsrError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {bsr_status_string(code)} ({code})")


class _Info(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32), ("num_qo_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32), ("causal", ctypes.c_int32),
        ("rope_theta", ctypes.c_float), ("sum_qo", ctypes.c_int64),
        ("active_tokens", ctypes.c_int64), ("num_decode_items", ctypes.c_int32),
        ("num_prefill_items", ctypes.c_int32), ("num_split_streams", ctypes.c_int32),
        ("num_partials", ctypes.c_int32), ("decode_ctas", ctypes.c_int32),
        ("decode_warps_per_cta", ctypes.c_int32), ("prefill_ctas", ctypes.c_int32),
        ("num_sms", ctypes.c_int32), ("workspace_bytes", ctypes.c_int64),
        ("upload_bytes", ctypes.c_int64),
        ("decode_imbalance", ctypes.c_double), ("prefill_imbalance", ctypes.c_double),
        ("kernels_per_run", ctypes.c_int32), ("window_left", ctypes.c_int32),
        ("kv_layout", ctypes.c_int32), ("kv_dtype", ctypes.c_int32),
    ]


def load(path: str | None = None):
    """Load the built library (raises if it is missing: there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or _build.lib_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build() "
                           "(block_sparse_kv_bsr_gb300._build.build())")
    lib = ctypes.CDLL(path)
    lib.bsr_attn_plan.restype = ctypes.c_int
    lib.bsr_attn_plan.argtypes = [_vp, _vp, _vp, ctypes.c_int32, ctypes.c_int32,
                                  ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _vp,
                                  ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _vp,
                                  ctypes.c_int32, ctypes.c_int32, ctypes.c_float, _vp,
                                  ctypes.POINTER(_vp)]
    lib.bsr_attn_plan_host.restype = ctypes.c_int
    lib.bsr_attn_plan_host.argtypes = [_vp, _vp, _vp, ctypes.c_int32, ctypes.c_int32,
                                       ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _vp,
                                       ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _vp,
                                       ctypes.c_int32, ctypes.c_int32, ctypes.c_float,
                                       ctypes.c_int32, ctypes.POINTER(_Info), _vp,
                                       ctypes.c_int64]
    lib.bsr_attn_run_kv8.restype = ctypes.c_int
    lib.bsr_attn_run_kv8.argtypes = [_vp, _vp, _vp, _vp, ctypes.c_float, ctypes.c_float,
                                     ctypes.c_float, ctypes.c_float, ctypes.c_int32, _vp,
                                     ctypes.c_int32, _vp, _vp]
    lib.bsr_attn_run.restype = ctypes.c_int
    lib.bsr_attn_run.argtypes = [_vp, _vp, _vp, _vp, ctypes.c_float, ctypes.c_float,
                                 ctypes.c_int32, _vp, ctypes.c_int32, _vp, _vp]
    lib.bsr_attn_run_host.restype = ctypes.c_int
    lib.bsr_attn_run_host.argtypes = [_vp, _vp, _vp, _vp, ctypes.c_float, ctypes.c_float,
                                      ctypes.c_float, ctypes.c_float, ctypes.c_int32, _vp,
                                      ctypes.c_int32, _vp, _vp]
    lib.bsr_merge_states.restype = ctypes.c_int
    lib.bsr_merge_states.argtypes = [_vp, _vp, _vp, _vp, ctypes.c_int64, ctypes.c_int32,
                                     ctypes.c_int32, ctypes.c_int32, _vp, _vp, _vp]
    lib.bsr_append_kv.restype = ctypes.c_int
    lib.bsr_append_kv.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_int32, ctypes.c_int64,
                                  ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                  ctypes.c_int32, _vp, _vp, _vp, _vp]
    lib.bsr_schedule_destroy.restype = None
    lib.bsr_schedule_destroy.argtypes = [_vp]
    lib.bsr_schedule_create.restype = ctypes.c_int
    lib.bsr_schedule_create.argtypes = [ctypes.c_int32, ctypes.POINTER(_vp)]
    lib.bsr_schedule_get_info.restype = ctypes.c_int
    lib.bsr_schedule_get_info.argtypes = [_vp, ctypes.POINTER(_Info)]
    lib.bsr_last_device_error.restype = ctypes.c_int
    lib.bsr_last_device_error.argtypes = [_vp]
    lib.bsr_selftest_bounded_wait.restype = ctypes.c_int
    lib.bsr_selftest_bounded_wait.argtypes = [_vp, ctypes.c_int64, _vp]
    lib.bsr_schedule_set_stage_timing.restype = ctypes.c_int
    lib.bsr_schedule_set_stage_timing.argtypes = [_vp, ctypes.c_int32]
    lib.bsr_schedule_stage_times.restype = ctypes.c_int
    lib.bsr_schedule_stage_times.argtypes = [_vp, ctypes.c_int32, ctypes.POINTER(ctypes.c_float)]
    lib.bsr_attn_decode_noalloc.restype = ctypes.c_int
    lib.bsr_attn_decode_noalloc.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_int32,
                                            ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                            ctypes.c_int32, ctypes.c_int32, ctypes.c_float, _vp,
                                            ctypes.c_int32, _vp, _vp, _vp]
    lib.bsr_attn_decode_noalloc_kv8.restype = ctypes.c_int
    lib.bsr_attn_decode_noalloc_kv8.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_int32,
                                                ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                                ctypes.c_int32, ctypes.c_int32, ctypes.c_float,
                                                ctypes.c_float, ctypes.c_float, _vp,
                                                ctypes.c_int32, _vp, _vp, _vp]
    lib.bsr_attn_decode_noalloc_ex.restype = ctypes.c_int
    lib.bsr_attn_decode_noalloc_ex.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_int32,
                                               ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                               ctypes.c_int32, ctypes.c_int32, ctypes.c_float,
                                               ctypes.c_int32, ctypes.c_float, ctypes.c_float,
                                               ctypes.c_int32, _vp, ctypes.c_int32, _vp, _vp,
                                               _vp]
    lib.bsr_status_string.restype = ctypes.c_char_p
    lib.bsr_status_string.argtypes = [ctypes.c_int]
    _lib = lib
    return lib


def bsr_status_string(code: int) -> str:
    return load().bsr_status_string(int(code)).decode()


BSR_KV_HND = 0
BSR_KV_NHD = 1


def _layout(kv_layout: str) -> int:
    """Page pool layout: "HND" [pages, Hk, P, D] or "NHD" [pages, P, Hk, D]."""
    if kv_layout not in ("HND", "NHD"):
        raise ValueError("kv_layout must be 'HND' or 'NHD'")
    return BSR_KV_NHD if kv_layout == "NHD" else BSR_KV_HND


def _kv_dtype(kv_dtype: str) -> int:
    """Cache element type: "bf16" (bsr_attn_run) or "e4m3" (bsr_attn_run_kv8)."""
    if kv_dtype not in ("bf16", "e4m3"):
        raise ValueError("kv_dtype must be 'bf16' or 'e4m3'")
    return 1 if kv_dtype == "e4m3" else 0


def _check(code: int, where: str):
    if code != BSR_OK:
        raise BsrError(code, where)


def _host_i32(x) -> np.ndarray:
    if hasattr(x, "detach"):
        if x.is_cuda:
            raise ValueError("plan reads host arrays: pass CPU tensors / numpy arrays")
        x = x.detach().numpy()
    return np.ascontiguousarray(x, dtype=np.int32)


def _host_i32_addr(x):
    """(object to keep alive, address or None) of a host int32 array; CPU int32 tensors and
    C-contiguous int32 numpy arrays are passed in place, anything else is converted."""
    if hasattr(x, "data_ptr"):
        if x.is_cuda:
            raise ValueError("plan reads host arrays: pass CPU tensors / numpy arrays")
        if x.dtype == _torch_int32() and x.is_contiguous():
            return x, (x.data_ptr() if x.numel() else None)
    elif isinstance(x, np.ndarray) and x.dtype == np.int32 and x.flags.c_contiguous:
        return x, (x.__array_interface__["data"][0] if x.size else None)
    a = _host_i32(x)
    return a, (a.__array_interface__["data"][0] if a.size else None)


def _torch_int32():
    import torch
    return torch.int32


def _stream_ptr(stream):
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


class Schedule:
    """Owns a ``bsr_schedule_t``; destroyed with :func:`bsr_schedule_destroy`."""

    def __init__(self, handle: int):
        self.handle = handle

    def info(self) -> dict:
        return bsr_schedule_get_info(self)

    def close(self):
        if self.handle:
            bsr_schedule_destroy(self)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def bsr_schedule_create(sm_budget: int = 0) -> Schedule:
    """An empty schedule whose plans use at most `sm_budget` SMs (0: all); plan into it
    with bsr_attn_plan(..., schedule=...)."""
    handle = _vp(None)
    _check(load().bsr_schedule_create(int(sm_budget), ctypes.byref(handle)), "bsr_schedule_create")
    return Schedule(handle.value)


def _plan_args(indptr, indices, last_page_len, qo_indptr):
    ip, ix, lp = _host_i32_addr(indptr), _host_i32_addr(indices), _host_i32_addr(last_page_len)
    qi = (None, None) if qo_indptr is None else _host_i32_addr(qo_indptr)
    keep = (ip[0], ix[0], lp[0], qi[0])
    return keep, (ip[1], ix[1], lp[1], qi[1]), len(ip[0]) - 1


def bsr_attn_plan(indptr, indices, last_page_len, *, num_qo_heads: int, num_kv_heads: int,
                  head_dim: int, page_size: int, num_pages: int, qo_indptr=None,
                  causal: bool = False, rope_theta: float = 0.0, window_left: int = 0,
                  page_pos=None, kv_layout: str = "HND", kv_dtype: str = "bf16", stream=None,
                  schedule: Schedule | None = None) -> Schedule:
    """Plan one batch from HOST page-table arrays; returns (or re-plans) a Schedule.
    kv_dtype: "bf16" for bsr_attn_run, "e4m3" for bsr_attn_run_kv8."""
    lib = load()
    keep, (ip, ix, lp, qi), batch = _plan_args(indptr, indices, last_page_len, qo_indptr)
    handle = _vp(schedule.handle if schedule is not None else None)
    pp = (None, None) if page_pos is None else _host_i32_addr(page_pos)
    code = lib.bsr_attn_plan(ip, ix, lp, batch, num_qo_heads, num_kv_heads, head_dim, page_size,
                             qi, int(num_pages), int(bool(causal)), int(window_left), pp[1],
                             _layout(kv_layout), _kv_dtype(kv_dtype), float(rope_theta),
                             _stream_ptr(stream),
                             ctypes.byref(handle))
    del keep
    _check(code, "bsr_attn_plan")
    if schedule is not None:
        schedule.handle = handle.value
        return schedule
    return Schedule(handle.value)


def bsr_attn_plan_host(indptr, indices, last_page_len, *, num_qo_heads: int, num_kv_heads: int,
                       head_dim: int, page_size: int, num_pages: int, num_sms: int,
                       qo_indptr=None, causal: bool = False, rope_theta: float = 0.0,
                       window_left: int = 0, page_pos=None, kv_layout: str = "HND",
                       kv_dtype: str = "bf16"):
    """Host-only planning for `num_sms` SMs: returns (info dict, units int32 [n, 8])."""
    lib = load()
    keep, (ip, ix, lp, qi), batch = _plan_args(indptr, indices, last_page_len, qo_indptr)
    pp = (None, None) if page_pos is None else _host_i32_addr(page_pos)
    args = [ip, ix, lp, batch, num_qo_heads, num_kv_heads, head_dim, page_size, qi,
            int(num_pages), int(bool(causal)), int(window_left), pp[1],
            _layout(kv_layout), _kv_dtype(kv_dtype), float(rope_theta), int(num_sms)]
    info = _Info()
    n = lib.bsr_attn_plan_host(*args, ctypes.byref(info), None, 0)
    if n < 0:
        raise BsrError(n, "bsr_attn_plan_host")
    units = np.zeros((max(n, 1), 8), dtype=np.int32)
    n2 = lib.bsr_attn_plan_host(*args, None, units.__array_interface__["data"][0], units.shape[0])
    del keep
    if n2 < 0:
        raise BsrError(n2, "bsr_attn_plan_host")
    return {name: getattr(info, name) for name, _ in _Info._fields_}, units[:n]


def bsr_attn_run(schedule: Schedule, q, k_pages, v_pages, *, sm_scale: float,
                 rope_theta: float = 0.0, causal: bool = False, out=None, lse=None,
                 out_dtype=None, want_lse: bool = True, stream=None):
    """Run a schedule; returns (out, lse).  out/lse are allocated here when not given."""
    import torch
    lib = load()
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype or torch.bfloat16, device=q.device)
    if lse is None and want_lse:
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    if out.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("out must be bf16 or fp32")
    dt = BSR_DTYPE_F32 if out.dtype == torch.float32 else BSR_DTYPE_BF16
    for t in (q, k_pages, v_pages):
        if t.dtype != torch.bfloat16:
            raise ValueError("q, k_pages, v_pages must be bf16")
    code = lib.bsr_attn_run(_vp(schedule.handle), _dptr(q), _dptr(k_pages), _dptr(v_pages),
                            float(sm_scale), float(rope_theta), int(bool(causal)), _dptr(out), dt,
                            _dptr(lse), _vp(_stream_ptr(stream)))
    _check(code, "bsr_attn_run")
    return out, lse


def _host_ptr(t):
    if t is None:
        return None
    if t.is_cuda:
        raise ValueError("expected a host (CPU) tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def bsr_attn_run_host(schedule: Schedule, q, k_pages, v_pages, *, sm_scale: float,
                      rope_theta: float = 0.0, causal: bool = False, k_scale: float = 1.0,
                      v_scale: float = 1.0, out=None, lse=None, out_dtype=None,
                      want_lse: bool = True, stream=None):
    """One step with HOST q / out / lse (pinned memory keeps the copies asynchronous):
    the upload, the run and the read-back are queued on `stream`; the host tensors hold
    the result once the stream has completed.  ``k_pages``/``v_pages`` are the device
    pools (bf16, or E4M3 codes with k_scale / v_scale for a schedule planned "e4m3")."""
    import torch
    lib = load()
    if q.dtype != torch.bfloat16:
        raise ValueError("q must be bf16")
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype or torch.bfloat16, pin_memory=True)
    if lse is None and want_lse:
        lse = torch.empty(q.shape[:2], dtype=torch.float32, pin_memory=True)
    if out.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("out must be bf16 or fp32")
    dt = BSR_DTYPE_F32 if out.dtype == torch.float32 else BSR_DTYPE_BF16
    code = lib.bsr_attn_run_host(_vp(schedule.handle), _host_ptr(q), _dptr(k_pages),
                                 _dptr(v_pages), float(k_scale), float(v_scale), float(sm_scale),
                                 float(rope_theta), int(bool(causal)), _host_ptr(out), dt,
                                 _host_ptr(lse), _vp(_stream_ptr(stream)))
    _check(code, "bsr_attn_run_host")
    return out, lse


def bsr_attn_run_kv8(schedule: Schedule, q, k_pages, v_pages, *, k_scale: float, v_scale: float,
                     sm_scale: float, rope_theta: float = 0.0, causal: bool = False, out=None,
                     lse=None, out_dtype=None, want_lse: bool = True, stream=None):
    """Run a schedule over an FP8 (E4M3) KV cache: ``k_pages``/``v_pages`` are uint8
    (or float8_e4m3fn) codes, the cached values ``k_scale * code`` / ``v_scale * code``."""
    import torch
    lib = load()
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype or torch.bfloat16, device=q.device)
    if lse is None and want_lse:
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    if out.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("out must be bf16 or fp32")
    if q.dtype != torch.bfloat16:
        raise ValueError("q must be bf16")
    for t in (k_pages, v_pages):
        if t.element_size() != 1:
            raise ValueError("k_pages, v_pages must hold one-byte E4M3 codes")
    dt = BSR_DTYPE_F32 if out.dtype == torch.float32 else BSR_DTYPE_BF16
    code = lib.bsr_attn_run_kv8(_vp(schedule.handle), _dptr(q), _dptr(k_pages), _dptr(v_pages),
                                float(k_scale), float(v_scale), float(sm_scale),
                                float(rope_theta), int(bool(causal)), _dptr(out), dt, _dptr(lse),
                                _vp(_stream_ptr(stream)))
    _check(code, "bsr_attn_run_kv8")
    return out, lse


def bsr_merge_states(o_a, lse_a, o_b, lse_b, *, o_out=None, lse_out=None, stream=None):
    """LSE-merge two attention states [rows, heads, D] (bf16 or fp32)."""
    import torch
    lib = load()
    if o_out is None:
        o_out = torch.empty_like(o_a)
    if lse_out is None:
        lse_out = torch.empty_like(lse_a)
    dt = BSR_DTYPE_F32 if o_a.dtype == torch.float32 else BSR_DTYPE_BF16
    rows, heads, D = o_a.shape
    code = lib.bsr_merge_states(_dptr(o_a), _dptr(lse_a), _dptr(o_b), _dptr(lse_b), rows, heads, D,
                                dt, _dptr(o_out), _dptr(lse_out), _vp(_stream_ptr(stream)))
    _check(code, "bsr_merge_states")
    return o_out, lse_out


def bsr_append_kv(k_new, v_new, append_indptr, indptr, indices, last_page_len, k_pages, v_pages,
                  *, kv_layout: str = "HND", device_status=None, stream=None):
    """Write new tokens' k/v into their pages (all arguments are device tensors); the
    pools are [pages, Hk, P, D] ("HND") or [pages, P, Hk, D] ("NHD")."""
    lib = load()
    if kv_layout == "NHD":
        num_pages, P, Hk, D = k_pages.shape
    else:
        num_pages, Hk, P, D = k_pages.shape
    code = lib.bsr_append_kv(_dptr(k_new), _dptr(v_new), _dptr(append_indptr), _dptr(indptr),
                             _dptr(indices), _dptr(last_page_len), len(indptr) - 1,
                             int(k_new.shape[0]), Hk, D, P, num_pages, _layout(kv_layout),
                             _dptr(k_pages), _dptr(v_pages), _dptr(device_status),
                             _vp(_stream_ptr(stream)))
    _check(code, "bsr_append_kv")


def bsr_schedule_destroy(schedule: Schedule):
    load().bsr_schedule_destroy(_vp(schedule.handle))
    schedule.handle = 0


def bsr_schedule_get_info(schedule: Schedule) -> dict:
    info = _Info()
    _check(load().bsr_schedule_get_info(_vp(schedule.handle), ctypes.byref(info)),
           "bsr_schedule_get_info")
    return {name: getattr(info, name) for name, _ in _Info._fields_}


def bsr_last_device_error(schedule: Schedule) -> int:
    code = load().bsr_last_device_error(_vp(schedule.handle))
    if code < 0:
        raise BsrError(code, "bsr_last_device_error")
    return code


def bsr_selftest_bounded_wait(device_status, limit_ns: int, stream=None):
    """Run one bounded wait that must run out (nothing arrives): sets bit 0 of the int32
    CUDA tensor `device_status` after `limit_ns`."""
    _check(load().bsr_selftest_bounded_wait(_vp(device_status.data_ptr()), int(limit_ns),
                                            _vp(_stream_ptr(stream))),
           "bsr_selftest_bounded_wait")


STAGES = ("decode", "prefill", "merge")


def bsr_schedule_set_stage_timing(schedule: Schedule, max_calls: int):
    """Record CUDA events around each kernel of the next runs (keeps the last max_calls)."""
    _check(load().bsr_schedule_set_stage_timing(_vp(schedule.handle), int(max_calls)),
           "bsr_schedule_set_stage_timing")


def bsr_schedule_stage_times(schedule: Schedule, call: int) -> dict:
    """Stage durations (ms) of kept run `call` (0 = oldest kept); absent stages omitted."""
    ms = (ctypes.c_float * len(STAGES))()
    code = load().bsr_schedule_stage_times(_vp(schedule.handle), int(call), ms)
    if code < 0:
        raise BsrError(code, "bsr_schedule_stage_times")
    return {name: float(ms[i]) for i, name in enumerate(STAGES) if ms[i] >= 0}


def bsr_attn_decode_noalloc(q, k_pages, v_pages, indptr, indices, last_page_len, *,
                            sm_scale: float, out, lse=None, device_status=None, stream=None):
    """Decode (one query per request) without any allocation inside the library.

    For callers that cannot allocate device memory at call time: every buffer,
    including ``out``, ``lse`` and the device page table, is the caller's; the
    library's scratch is a fixed static device array shared by all calls on a
    device (serialize calls on one stream).
    """
    import torch
    lib = load()
    num_pages, Hk, P, D = k_pages.shape
    batch, Hq = q.shape[0], q.shape[1]
    dt = BSR_DTYPE_F32 if out.dtype == torch.float32 else BSR_DTYPE_BF16
    code = lib.bsr_attn_decode_noalloc(_dptr(q), _dptr(k_pages), _dptr(v_pages), _dptr(indptr),
                                       _dptr(indices), _dptr(last_page_len), batch, Hq, Hk, D, P,
                                       num_pages, float(sm_scale), _dptr(out), dt, _dptr(lse),
                                       _dptr(device_status), _vp(_stream_ptr(stream)))
    _check(code, "bsr_attn_decode_noalloc")
    return out, lse


def bsr_attn_decode_noalloc_kv8(q, k_pages, v_pages, indptr, indices, last_page_len, *,
                                sm_scale: float, k_scale: float, v_scale: float, out, lse=None,
                                device_status=None, stream=None):
    """bsr_attn_decode_noalloc over an FP8 (E4M3) cache: uint8 (or float8_e4m3fn) codes,
    the cached values ``k_scale * code`` / ``v_scale * code``."""
    import torch
    lib = load()
    num_pages, Hk, P, D = k_pages.shape
    batch, Hq = q.shape[0], q.shape[1]
    dt = BSR_DTYPE_F32 if out.dtype == torch.float32 else BSR_DTYPE_BF16
    code = lib.bsr_attn_decode_noalloc_kv8(_dptr(q), _dptr(k_pages), _dptr(v_pages),
                                           _dptr(indptr), _dptr(indices), _dptr(last_page_len),
                                           batch, Hq, Hk, D, P, num_pages, float(sm_scale),
                                           float(k_scale), float(v_scale), _dptr(out), dt,
                                           _dptr(lse), _dptr(device_status),
                                           _vp(_stream_ptr(stream)))
    _check(code, "bsr_attn_decode_noalloc_kv8")
    return out, lse


def bsr_attn_decode_noalloc_ex(q, k_pages, v_pages, indptr, indices, last_page_len, *,
                               sm_scale: float, out, kv_dtype: str = "bf16", k_scale: float = 1.0,
                               v_scale: float = 1.0, window_left: int = 0, lse=None,
                               device_status=None, stream=None):
    """No-allocation decode with the cache element type ("bf16" or "e4m3", the latter with
    k_scale / v_scale) and an optional sliding window of ``window_left`` keys."""
    import torch
    lib = load()
    num_pages, Hk, P, D = k_pages.shape
    batch, Hq = q.shape[0], q.shape[1]
    kd = {"bf16": 0, "e4m3": 1}[kv_dtype]
    dt = BSR_DTYPE_F32 if out.dtype == torch.float32 else BSR_DTYPE_BF16
    code = lib.bsr_attn_decode_noalloc_ex(_dptr(q), _dptr(k_pages), _dptr(v_pages),
                                          _dptr(indptr), _dptr(indices), _dptr(last_page_len),
                                          batch, Hq, Hk, D, P, num_pages, float(sm_scale), kd,
                                          float(k_scale), float(v_scale), int(window_left),
                                          _dptr(out), dt, _dptr(lse), _dptr(device_status),
                                          _vp(_stream_ptr(stream)))
    _check(code, "bsr_attn_decode_noalloc_ex")
    return out, lse
