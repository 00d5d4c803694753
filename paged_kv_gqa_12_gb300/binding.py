"""Thin ctypes binding of the C ABI in ``include/pa.h``.

Argument marshalling only: every step of the computation runs in the CUDA
library.  Tensors are torch tensors on the current CUDA device; their data
pointers and element strides are passed through unchanged.  If the library
has not been built, loading raises -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

PA_OK = 0
PA_ERR_INVALID_ARG = 1
PA_ERR_UNSUPPORTED = 2
PA_ERR_SCRATCH_TOO_SMALL = 3
PA_ERR_CUDA = 4
PA_ERR_DEVICE = 5

# bits of the device error code pa_check reports (pa_device_code)
DEVICE_WAIT_TIMEOUT = 1
DEVICE_WORK_OVERFLOW = 2
DEVICE_CAPACITY = 4
DEVICE_PAGE_ID = 8

# bytes of the scratch header (error word, then split-arrival counters) at
# the start of every scratch workspace
SCRATCH_HEADER_BYTES = 65536
# (request, kv head group) pairs a plan may have for its last split to merge
MERGE_COUNTERS = (SCRATCH_HEADER_BYTES - 256) // 4

MODE_DECODE = 0
MODE_EXTEND = 1
MODE_VERIFY = 2
KV_BF16 = 0
KV_FP8_E4M3 = 1

EXPORTED_SYMBOLS = ("pa_plan", "pa_decode", "pa_extend", "pa_scratch_init", "pa_check",
                    "pa_status_string", "pa_version", "pa_decode_static_scratch", "pa_append_kv",
                    "pa_debug_wait_expiry")


class PaShape(ctypes.Structure):
    _fields_ = [
        ("mode", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("kv_dtype", ctypes.c_int32),
        ("max_batch", ctypes.c_int32),
        ("max_pages_per_seq", ctypes.c_int32),
        ("max_total_q", ctypes.c_int32),
        ("window", ctypes.c_int32),
        ("has_sinks", ctypes.c_int32),
        ("soft_cap", ctypes.c_float),
        ("num_splits", ctypes.c_int32),
        ("num_sms", ctypes.c_int32),
        ("q_len", ctypes.c_int32),
    ]


class PaPlan(ctypes.Structure):
    _fields_ = [
        ("shape", PaShape),
        ("tile_tokens", ctypes.c_int32),
        ("split_tiles", ctypes.c_int32),
        ("max_splits", ctypes.c_int32),
        ("stages", ctypes.c_int32),
        ("warps", ctypes.c_int32),
        ("bt_cache", ctypes.c_int32),
        ("smem_bytes", ctypes.c_int32),
        ("grid", ctypes.c_int32 * 3),
        ("scratch_bytes", ctypes.c_int64),
        ("launches", ctypes.c_int32),
        ("kv_copy", ctypes.c_int32),
        ("split_merge", ctypes.c_int32),
        ("reserved", ctypes.c_int32 * 5),
    ]


class PaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the CUDA library (build it first with ``paged_kv_gqa_12_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or _build.LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built: {path} is missing "
                           "(run paged_kv_gqa_12_gb300.build.build())")
    L = ctypes.CDLL(path)
    vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    L.pa_plan.argtypes = [ctypes.POINTER(PaShape), vp, i32, ctypes.POINTER(PaPlan)]
    L.pa_plan.restype = ctypes.c_int
    L.pa_decode.argtypes = [ctypes.POINTER(PaPlan), vp, i64, i64, vp, vp, i64, i64, i64, i32, vp, i64,
                            vp, i32, f32, vp, f32, f32, vp, vp, vp, i64, i64, vp, vp, i64, vp]
    L.pa_decode.restype = ctypes.c_int
    L.pa_extend.argtypes = [ctypes.POINTER(PaPlan), vp, i64, i64, vp, vp, i64, i64, i64, i32, vp, i64,
                            vp, vp, i32, i32, f32, vp, f32, f32, vp, vp, vp, i64, i64, vp, vp, i64, vp]
    L.pa_extend.restype = ctypes.c_int
    L.pa_decode_static_scratch.argtypes = [ctypes.POINTER(PaPlan), vp, i64, i64, vp, vp, i64, i64, i64, i32,
                                           vp, i64, vp, i32, f32, vp, f32, f32, vp, i64, i64, vp, vp]
    L.pa_decode_static_scratch.restype = ctypes.c_int
    L.pa_append_kv.argtypes = [vp, vp, i64, i64, vp, vp, i64, i64, i64, i32, i32, i32, i32, i32, vp, i32, f32, f32,
                               vp, vp]
    L.pa_append_kv.restype = ctypes.c_int
    L.pa_debug_wait_expiry.argtypes = [vp, i32, i64, vp]
    L.pa_debug_wait_expiry.restype = ctypes.c_int
    L.pa_scratch_init.argtypes = [vp, vp]
    L.pa_scratch_init.restype = ctypes.c_int
    L.pa_check.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint32)]
    L.pa_check.restype = ctypes.c_int
    L.pa_status_string.argtypes = [ctypes.c_int]
    L.pa_status_string.restype = ctypes.c_char_p
    L.pa_version.argtypes = []
    L.pa_version.restype = i32
    _lib = L
    return L


def status_string(status: int) -> str:
    return load().pa_status_string(int(status)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status: int, where: str):
    if status != PA_OK:
        raise PaError(status, where)


def plan(*, mode: int, num_q_heads: int, num_kv_heads: int, head_dim: int, page_size: int,
         kv_dtype: int = KV_BF16, max_batch: int, max_pages_per_seq: int, max_total_q: int = 0,
         window: int = 0, has_sinks: bool = False, soft_cap: float = 0.0, num_splits: int = 0,
         num_sms: int = 0, q_len: int = 0, host_seq_lens=None) -> PaPlan:
    """pa_plan.  ``host_seq_lens``: optional host int32 sequence of lengths."""
    s = PaShape(mode=mode, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
                page_size=page_size, kv_dtype=kv_dtype, max_batch=max_batch,
                max_pages_per_seq=max_pages_per_seq, max_total_q=max_total_q, window=window,
                has_sinks=1 if has_sinks else 0, soft_cap=soft_cap, num_splits=num_splits, num_sms=num_sms,
                q_len=q_len)
    p = PaPlan()
    lens_arr, n = None, 0
    if host_seq_lens is not None:
        vals = [int(x) for x in host_seq_lens]
        n = len(vals)
        lens_arr = (ctypes.c_int32 * max(n, 1))(*vals)
    _check(load().pa_plan(ctypes.byref(s), lens_arr, n, ctypes.byref(p)), "pa_plan")
    return p


def _kv_strides(k_cache, v_cache):
    if tuple(k_cache.stride()) != tuple(v_cache.stride()) or k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache must share shape and strides")
    if k_cache.dim() != 4 or k_cache.stride(3) != 1:
        raise ValueError("caches must be [pages, page_size, kv_heads, head_dim] with contiguous head_dim")
    return k_cache.stride(0), k_cache.stride(1), k_cache.stride(2)


def decode(p: PaPlan, q, k_cache, v_cache, block_table, seq_lens, *, scale: float, out, lse=None,
           sinks=None, k_scale: float = 1.0, v_scale: float = 1.0, k_scales=None, v_scales=None, scratch,
           stream=None):
    """pa_decode on torch tensors (q/out [B, Hq, D] bf16; caches bf16 or uint8 e4m3;
    k_scales / v_scales: optional device fp32 [B] per-request descales)."""
    sp, st, sh = _kv_strides(k_cache, v_cache)
    status = load().pa_decode(
        ctypes.byref(p), _ptr(q), q.stride(0), q.stride(1), _ptr(k_cache), _ptr(v_cache), sp, st, sh,
        k_cache.shape[0], _ptr(block_table), block_table.stride(0), _ptr(seq_lens), seq_lens.shape[0],
        float(scale), _ptr(sinks), float(k_scale), float(v_scale), _ptr(k_scales), _ptr(v_scales), _ptr(out),
        out.stride(0), out.stride(1), _ptr(lse), _ptr(scratch), scratch.numel() * scratch.element_size(),
        _stream(stream))
    _check(status, "pa_decode")


def extend(p: PaPlan, q, k_cache, v_cache, block_table, seq_lens, query_start_loc, *, scale: float, out,
           lse=None, sinks=None, k_scale: float = 1.0, v_scale: float = 1.0, k_scales=None, v_scales=None,
           scratch, stream=None):
    """pa_extend on torch tensors (q/out [T, Hq, D] bf16; k_scales / v_scales:
    optional device fp32 [B] per-request descales)."""
    sp, st, sh = _kv_strides(k_cache, v_cache)
    status = load().pa_extend(
        ctypes.byref(p), _ptr(q), q.stride(0), q.stride(1), _ptr(k_cache), _ptr(v_cache), sp, st, sh,
        k_cache.shape[0], _ptr(block_table), block_table.stride(0), _ptr(seq_lens), _ptr(query_start_loc),
        seq_lens.shape[0], q.shape[0], float(scale), _ptr(sinks), float(k_scale), float(v_scale), _ptr(k_scales),
        _ptr(v_scales), _ptr(out), out.stride(0), out.stride(1), _ptr(lse), _ptr(scratch),
        scratch.numel() * scratch.element_size(), _stream(stream))
    _check(status, "pa_extend")


def decode_static_scratch(p: PaPlan, q, k_cache, v_cache, block_table, seq_lens, *, scale: float, out,
                          lse=None, sinks=None, k_scale: float = 1.0, v_scale: float = 1.0, stream=None):
    """pa_decode_static_scratch: decode for callers that cannot allocate a
    workspace; the library's own fixed 16 MiB device array is used instead
    (calls on one device must not overlap)."""
    sp, st, sh = _kv_strides(k_cache, v_cache)
    status = load().pa_decode_static_scratch(
        ctypes.byref(p), _ptr(q), q.stride(0), q.stride(1), _ptr(k_cache), _ptr(v_cache), sp, st, sh,
        k_cache.shape[0], _ptr(block_table), block_table.stride(0), _ptr(seq_lens), seq_lens.shape[0],
        float(scale), _ptr(sinks), float(k_scale), float(v_scale), _ptr(out), out.stride(0), out.stride(1),
        _ptr(lse), _stream(stream))
    _check(status, "pa_decode_static_scratch")


def append_kv(k_new, v_new, k_cache, v_cache, slot_mapping, *, kv_dtype: int = KV_BF16, k_scale: float = 1.0,
              v_scale: float = 1.0, scratch=None, stream=None):
    """pa_append_kv: write new tokens' K/V (bf16 [T, Hkv, D]) into the paged caches at slot_mapping (int64)."""
    sp, st, sh = _kv_strides(k_cache, v_cache)
    if tuple(k_new.stride()) != tuple(v_new.stride()) or k_new.shape != v_new.shape:
        raise ValueError("k_new and v_new must share shape and strides")
    status = load().pa_append_kv(
        _ptr(k_new), _ptr(v_new), k_new.stride(0), k_new.stride(1), _ptr(k_cache), _ptr(v_cache), sp, st, sh,
        k_cache.shape[0], k_cache.shape[1], k_cache.shape[2], k_cache.shape[3], int(kv_dtype), _ptr(slot_mapping),
        k_new.shape[0], float(k_scale), float(v_scale), _ptr(scratch), _stream(stream))
    _check(status, "pa_append_kv")


def debug_wait_expiry(scratch, which: int, limit_ns: int, stream=None):
    """pa_debug_wait_expiry: run one bounded device wait out on purpose (test hook)."""
    _check(load().pa_debug_wait_expiry(_ptr(scratch), int(which), int(limit_ns), _stream(stream)),
           "pa_debug_wait_expiry")


def scratch_init(scratch, stream=None):
    _check(load().pa_scratch_init(_ptr(scratch), _stream(stream)), "pa_scratch_init")


def check(scratch, stream=None) -> int:
    """pa_check: synchronises and returns the device error code (0 = none)."""
    code = ctypes.c_uint32(0)
    status = load().pa_check(_ptr(scratch), _stream(stream), ctypes.byref(code))
    if status not in (PA_OK, PA_ERR_DEVICE):
        raise PaError(status, "pa_check")
    return int(code.value)


def alloc_scratch(p: PaPlan, device=None):
    """Allocate a scratch workspace (torch uint8, 256-byte aligned) for a plan
    and zero its error header."""
    n = int(p.scratch_bytes)
    buf = torch.empty(n + 256, dtype=torch.uint8, device=device or "cuda")
    off = (-buf.data_ptr()) % 256
    s = buf[off:off + n]
    scratch_init(s)
    return s
