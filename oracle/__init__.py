"""Test infrastructure -- NOT part of the product.

ctypes wrapper around ``oracle.cpp``: the plain fp64 CPU oracle of paged-KV
grouped-query attention (decode and prefix-prefill/extend).  Only the tests,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
this package.  It shares no code with the CUDA library and imports nothing
from it.

Every function of the oracle is pinned by ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile liboracle.so with the host compiler.

    ``-ffp-contract=off`` keeps every multiply and add separately rounded, so
    the oracle gives bit-identical results on x86-64 and aarch64 hosts.
    """
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-shared", "-fPIC", "-pthread", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Problem(ctypes.Structure):
    _fields_ = [
        ("mode", ctypes.c_int),
        ("batch", ctypes.c_int),
        ("num_q_heads", ctypes.c_int),
        ("num_kv_heads", ctypes.c_int),
        ("head_dim", ctypes.c_int),
        ("page_size", ctypes.c_int),
        ("num_pages", ctypes.c_int),
        ("q", ctypes.c_void_p),
        ("q_stride_row", ctypes.c_int64),
        ("q_stride_head", ctypes.c_int64),
        ("k_cache", ctypes.c_void_p),
        ("v_cache", ctypes.c_void_p),
        ("kv_fp8", ctypes.c_int),
        ("kv_stride_page", ctypes.c_int64),
        ("kv_stride_tok", ctypes.c_int64),
        ("kv_stride_head", ctypes.c_int64),
        ("block_table", ctypes.c_void_p),
        ("bt_stride", ctypes.c_int64),
        ("seq_lens", ctypes.c_void_p),
        ("query_start_loc", ctypes.c_void_p),
        ("scale", ctypes.c_double),
        ("window", ctypes.c_int),
        ("soft_cap", ctypes.c_double),
        ("sinks", ctypes.c_void_p),
        ("k_scale", ctypes.c_float),
        ("v_scale", ctypes.c_float),
        ("k_scales", ctypes.c_void_p),
        ("v_scales", ctypes.c_void_p),
        ("rows", ctypes.c_void_p),
        ("num_rows", ctypes.c_int),
        ("out", ctypes.c_void_p),
        ("lse", ctypes.c_void_p),
        ("num_threads", ctypes.c_int),
    ]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            L.oracle_attention.argtypes = [ctypes.POINTER(_Problem)]
            L.oracle_attention.restype = ctypes.c_int
            L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            L.oracle_bf16_to_double.restype = ctypes.c_double
            L.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
            L.oracle_e4m3_to_double.restype = ctypes.c_double
            L.oracle_fp8_dequant.argtypes = [ctypes.c_uint8, ctypes.c_float]
            L.oracle_fp8_dequant.restype = ctypes.c_double
            L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
            L.oracle_e4m3_encode.restype = ctypes.c_uint8
            vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            L.oracle_append_kv.argtypes = [vp, vp, i64, i64, vp, vp, i64, i64, i64, i32, i32, vp, i32, i32, i32,
                                           i32, ctypes.c_float, ctypes.c_float]
            L.oracle_append_kv.restype = ctypes.c_int
            _lib = L
    return _lib


def bf16_to_double(bits: int) -> float:
    return lib().oracle_bf16_to_double(int(bits))


def e4m3_to_double(code: int) -> float:
    return lib().oracle_e4m3_to_double(int(code))


def fp8_dequant(code: int, scale: float) -> float:
    return lib().oracle_fp8_dequant(int(code), float(scale))


def e4m3_encode(y: float) -> int:
    return int(lib().oracle_e4m3_encode(float(y)))


def append_kv(k_new: np.ndarray, v_new: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
              slot_mapping: np.ndarray, k_scale: float = 1.0, v_scale: float = 1.0) -> None:
    """Write new tokens' K/V (uint16 bf16 bits [T, Hkv, D]) into the caches
    ([pages, page_size, Hkv, D], uint16 or uint8 e4m3), in place."""
    L = lib()
    assert k_new.dtype == np.uint16 and v_new.shape == k_new.shape and k_new.strides == v_new.strides
    assert k_cache.strides == v_cache.strides and k_cache.dtype == v_cache.dtype
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    ns = _elem_strides(k_new)
    ks = _elem_strides(k_cache)
    rc = L.oracle_append_kv(k_new.ctypes.data, v_new.ctypes.data, ns[0], ns[1], k_cache.ctypes.data,
                            v_cache.ctypes.data, ks[0], ks[1], ks[2], k_cache.shape[0], k_cache.shape[1],
                            sm.ctypes.data, sm.shape[0], k_new.shape[1], k_new.shape[2],
                            1 if k_cache.dtype == np.uint8 else 0, float(k_scale), float(v_scale))
    if rc != 0:
        raise RuntimeError(f"oracle_append_kv failed with code {rc}")


def _elem_strides(a: np.ndarray):
    return [s // a.itemsize for s in a.strides]


def attention(p, rows=None, num_threads: int | None = None):
    """Evaluate the oracle on a problem from the seeded input generators.

    ``p`` carries numpy arrays: q (uint16 bf16 bits [T, Hq, D]), k_cache /
    v_cache ([pages, page_size, Hkv, D], uint16 bf16 bits or uint8 e4m3
    codes, any strides), block_table, seq_lens, query_start_loc (extend) and
    the scalar options; optional ``k_scales`` / ``v_scales`` ([batch] fp32)
    are per-request e4m3 descales that replace ``k_scale`` / ``v_scale``.
    ``rows`` optionally selects query rows.  Returns (out [n, Hq, D] float64,
    lse [n, Hq] float64).
    """
    L = lib()
    q = p.q
    assert q.dtype == np.uint16 and q.ndim == 3 and q.strides[2] == 2
    kc, vc = p.k_cache, p.v_cache
    assert kc.shape == vc.shape and kc.strides == vc.strides and kc.dtype == vc.dtype
    fp8 = kc.dtype == np.uint8
    ks = _elem_strides(kc)
    assert ks[3] == 1
    bt = np.ascontiguousarray(p.block_table, dtype=np.int32)
    sl = np.ascontiguousarray(p.seq_lens, dtype=np.int32)
    qsl = None if p.query_start_loc is None else np.ascontiguousarray(p.query_start_loc, dtype=np.int32)
    sinks = None if p.sinks is None else np.ascontiguousarray(p.sinks, dtype=np.float32)
    B = int(sl.shape[0])
    kss = getattr(p, "k_scales", None)
    vss = getattr(p, "v_scales", None)
    kss = None if kss is None else np.ascontiguousarray(kss, dtype=np.float32)
    vss = None if vss is None else np.ascontiguousarray(vss, dtype=np.float32)
    assert kss is None or kss.shape == (B,)
    assert vss is None or vss.shape == (B,)
    T = q.shape[0]
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    n = T if r is None else int(r.shape[0])
    Hq, D = q.shape[1], q.shape[2]
    out = np.zeros((n, Hq, D), np.float64)
    lse = np.zeros((n, Hq), np.float64)
    qs = _elem_strides(q)
    prob = _Problem(
        mode=0 if p.mode == "decode" else 1,
        batch=B, num_q_heads=Hq, num_kv_heads=kc.shape[2], head_dim=D,
        page_size=kc.shape[1], num_pages=kc.shape[0],
        q=q.ctypes.data, q_stride_row=qs[0], q_stride_head=qs[1],
        k_cache=kc.ctypes.data, v_cache=vc.ctypes.data, kv_fp8=1 if fp8 else 0,
        kv_stride_page=ks[0], kv_stride_tok=ks[1], kv_stride_head=ks[2],
        block_table=bt.ctypes.data, bt_stride=bt.shape[1],
        seq_lens=sl.ctypes.data,
        query_start_loc=None if qsl is None else qsl.ctypes.data,
        scale=float(p.scale), window=int(p.window), soft_cap=float(p.soft_cap),
        sinks=None if sinks is None else sinks.ctypes.data,
        k_scale=float(p.k_scale), v_scale=float(p.v_scale),
        k_scales=None if kss is None else kss.ctypes.data, v_scales=None if vss is None else vss.ctypes.data,
        rows=None if r is None else r.ctypes.data, num_rows=n,
        out=out.ctypes.data, lse=lse.ctypes.data,
        num_threads=int(num_threads or os.cpu_count() or 1),
    )
    rc = L.oracle_attention(ctypes.byref(prob))
    if rc != 0:
        raise RuntimeError(f"oracle_attention failed with code {rc}")
    return out, lse
