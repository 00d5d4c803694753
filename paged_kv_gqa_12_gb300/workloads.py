"""Seeded synthetic inputs for paged-KV grouped-query attention.

This module only builds inputs: sequence lengths, a shuffled page pool with
per-request block tables, bf16 queries and a bf16 or fp8-e4m3 KV cache.  It
holds none of the attention arithmetic, and both the CUDA path and the CPU
oracle consume the same arrays it returns.

Layout follows the paged cache views of the b12x backend page
("vllm/v1/attention/backends/b12x", ``_kv_cache_views``): K and V are each
``[num_pages, page_size, num_kv_heads, head_dim]``, either as two separate
pools or as the two halves of one ``[num_pages, 2, page_size, Hkv*D]`` tensor.
Token ``t`` of request ``b`` is written to page ``block_table[b, t // ps]``,
slot ``t % ps`` -- the cache-append side of the map the decode page
("triton_decode_attention.py", ``_fwd_grouped_kernel_stage1``) reads.

Poisoning: every cache slot no query can attend to (pool pages no request
owns, slots past a sequence's end, pages wholly before a sliding window) holds
NaN, and unused block-table entries hold INT32_MAX, so a kernel that reads
outside the attended set produces NaN instead of a plausible number.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np
import torch

BT_SENTINEL = np.iinfo(np.int32).max
BF16_NAN = 0x7FC0
E4M3_NAN = 0x7F
E4M3_MAX = 448.0


@dataclass
class Problem:
    mode: str                      # "decode" or "extend"
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    kv_dtype: str                  # "bf16" or "fp8_e4m3"
    q: np.ndarray                  # uint16 bf16 bits [T, Hq, D]
    k_cache: np.ndarray            # [P, ps, Hkv, D] uint16 (bf16) / uint8 (e4m3)
    v_cache: np.ndarray
    block_table: np.ndarray        # int32 [B, W]
    seq_lens: np.ndarray           # int32 [B], cached + new tokens
    query_start_loc: np.ndarray | None  # int32 [B+1] (extend)
    scale: float
    window: int = 0
    soft_cap: float = 0.0
    sinks: np.ndarray | None = None     # float32 [Hq]
    k_scale: float = 1.0
    v_scale: float = 1.0
    k_scales: np.ndarray | None = None    # float32 [B]: per-request e4m3 descales (replace k_scale)
    v_scales: np.ndarray | None = None
    kv_storage: np.ndarray | None = None  # backing array when K/V are views
    logical_k: list | None = field(default=None, repr=False)  # per request [L_b, Hkv, D]
    logical_v: list | None = field(default=None, repr=False)
    name: str = ""

    @property
    def batch(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def num_pages(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def num_rows(self) -> int:
        return int(self.q.shape[0])

    def query_lens(self) -> np.ndarray:
        if self.mode == "decode":
            return np.ones(self.batch, np.int32)
        return np.diff(self.query_start_loc).astype(np.int32)


def _to_bf16_bits(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _to_e4m3_codes(x: np.ndarray, scale: float) -> np.ndarray:
    # Generator-side quantisation of the synthetic cache: x / scale, saturated
    # to the finite e4m3 range, rounded to nearest even by torch.
    y = np.clip(np.asarray(x, np.float32) / np.float32(scale), -E4M3_MAX, E4M3_MAX)
    t = torch.from_numpy(np.ascontiguousarray(y)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def build_problem(mode: str, *, num_q_heads: int, num_kv_heads: int, head_dim: int,
                  page_size: int, seq_lens, query_lens=None, kv_dtype: str = "bf16",
                  scale: float | None = None, window: int = 0, soft_cap: float = 0.0,
                  sinks: bool = False, k_scale: float = 1.0, v_scale: float = 1.0,
                  k_scales=None, v_scales=None,
                  pool_extra: float = 0.10, pool_pages: int | None = None,
                  bt_width: int | None = None, seed: int = 0, layout: str = "separate",
                  poison: bool = True, keep_logical: bool = False, threads: int | None = None,
                  q_values=None, name: str = "") -> Problem:
    """Build one seeded problem.

    ``seq_lens[b]`` counts every key of request b (for extend: cached context
    plus the new tokens, which are already in the pages).  ``query_lens``
    (extend only) gives the new tokens per request.  ``q_values`` (optional,
    float32 [T, Hq, D]) replaces the random queries; it is rounded to bf16.
    ``k_scales`` / ``v_scales`` (e4m3 only, [B]) quantise each request's keys /
    values with its own scale and are kept as per-request descales.
    """
    assert mode in ("decode", "extend")
    assert kv_dtype in ("bf16", "fp8_e4m3")
    assert layout in ("separate", "interleaved")
    rng = np.random.default_rng(seed)
    sl = np.asarray(seq_lens, dtype=np.int64)
    B = int(sl.shape[0])
    Hq, Hkv, D, ps = num_q_heads, num_kv_heads, head_dim, page_size
    if mode == "extend":
        ql = np.asarray(query_lens, dtype=np.int64)
        assert ql.shape == (B,) and np.all(ql >= 0) and np.all(ql <= sl)
        qsl = np.zeros(B + 1, np.int64)
        qsl[1:] = np.cumsum(ql)
    else:
        ql = np.ones(B, np.int64)
        qsl = None
    if scale is None:
        scale = head_dim ** -0.5

    # Page pool: a seeded permutation dealt out to the requests in order.
    n_pages = [(int(L) + ps - 1) // ps for L in sl]
    need = int(sum(n_pages))
    if pool_pages is None:
        pool_pages = max(1, int(math.ceil(need * (1.0 + pool_extra))))
    assert pool_pages >= need, "page pool too small"
    perm = rng.permutation(pool_pages).astype(np.int32)
    W = bt_width if bt_width is not None else max(1, max(n_pages, default=1))
    assert W >= max(n_pages, default=0)
    bt = np.full((B, W), BT_SENTINEL, np.int32)
    off = 0
    for b in range(B):
        bt[b, :n_pages[b]] = perm[off:off + n_pages[b]]
        off += n_pages[b]

    # KV storage, poisoned.
    fp8 = kv_dtype == "fp8_e4m3"
    kss = None if k_scales is None else np.asarray(k_scales, np.float32).reshape(-1)
    vss = None if v_scales is None else np.asarray(v_scales, np.float32).reshape(-1)
    assert (kss is None and vss is None) or fp8, "per-request scales apply to an e4m3 cache"
    assert kss is None or kss.shape == (B,)
    assert vss is None or vss.shape == (B,)
    dt = np.uint8 if fp8 else np.uint16
    fill = (E4M3_NAN if fp8 else BF16_NAN) if poison else 0
    if layout == "separate":
        k_cache = np.full((pool_pages, ps, Hkv, D), fill, dt)
        v_cache = np.full((pool_pages, ps, Hkv, D), fill, dt)
        storage = None
    else:
        storage = np.full((pool_pages, 2, ps, Hkv * D), fill, dt)
        k_cache = storage[:, 0].reshape(pool_pages, ps, Hkv, D)
        v_cache = storage[:, 1].reshape(pool_pages, ps, Hkv, D)
        assert np.shares_memory(k_cache, storage) and np.shares_memory(v_cache, storage)

    # First key any query of request b can see: the sliding window keeps key j
    # for query position p iff p - j < window.
    def first_reachable(b):
        if window <= 0:
            return 0
        first_q = int(sl[b]) - int(ql[b])          # position of the first query
        if mode == "decode":
            first_q = int(sl[b]) - 1
        return max(0, first_q - window + 1)

    children = np.random.SeedSequence(seed).spawn(B + 1)
    logical_k = [None] * B if keep_logical else None
    logical_v = [None] * B if keep_logical else None

    def fill_request(b):
        L = int(sl[b])
        if L == 0:
            return
        g = np.random.default_rng(children[b])
        t0 = (first_reachable(b) // ps) * ps      # whole pages from the window start
        n = L - t0
        kx = g.standard_normal((n, Hkv, D), dtype=np.float32)
        vx = g.standard_normal((n, Hkv, D), dtype=np.float32)
        if fp8:
            ksc = k_scale if kss is None else float(kss[b])
            vsc = v_scale if vss is None else float(vss[b])
            kq, vq = _to_e4m3_codes(kx, ksc), _to_e4m3_codes(vx, vsc)
        else:
            kq, vq = _to_bf16_bits(kx), _to_bf16_bits(vx)
        tok = np.arange(t0, L)
        pages = bt[b, tok // ps]
        slots = tok % ps
        k_cache[pages, slots] = kq
        v_cache[pages, slots] = vq
        if keep_logical:
            lk = np.full((L, Hkv, D), fill, dt)
            lv = np.full((L, Hkv, D), fill, dt)
            lk[t0:] = kq
            lv[t0:] = vq
            logical_k[b], logical_v[b] = lk, lv

    nthreads = threads or min(16, os.cpu_count() or 1)
    if B > 1 and nthreads > 1:
        with ThreadPoolExecutor(nthreads) as ex:
            list(ex.map(fill_request, range(B)))
    else:
        for b in range(B):
            fill_request(b)

    T = int(ql.sum())
    if q_values is None:
        gq = np.random.default_rng(children[B])
        qf = gq.standard_normal((T, Hq, D), dtype=np.float32)
    else:
        qf = np.asarray(q_values, np.float32)
        assert qf.shape == (T, Hq, D)
    q = _to_bf16_bits(qf)
    sk = rng.standard_normal(Hq).astype(np.float32) if sinks else None

    return Problem(
        mode=mode, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=ps,
        kv_dtype=kv_dtype, q=q, k_cache=k_cache, v_cache=v_cache, block_table=bt,
        seq_lens=sl.astype(np.int32),
        query_start_loc=None if qsl is None else qsl.astype(np.int32),
        scale=float(scale), window=int(window), soft_cap=float(soft_cap), sinks=sk,
        k_scale=float(k_scale), v_scale=float(v_scale), k_scales=kss, v_scales=vss, kv_storage=storage,
        logical_k=logical_k, logical_v=logical_v, name=name)


# ---- the five benchmark workloads --------------------------------------------

WORKLOADS = {
    "decode_tiny": "decode-tiny B4 Hq8 Hkv2 D64 ps16 S4",
    "decode_llama3_8b": "decode Llama-3-8B-shaped B64 Hq32 Hkv8 D128 ps16 bf16 L~U[512,8192]",
    "decode_e4m3_window": "decode fp8-e4m3 B128 Hq64 Hkv8 D64 ps64 window1024 sinks L~logU[1024,32768]",
    "prefill": "extend B8 Hq32 Hkv8 D128 ps16 ctx~U[0,4096] q~U[1,2048]",
    "decode_softcap_d256": "decode softcap50 window4096 B256 Hq16 Hkv8 D256 ps32 L~lognormal(2048,1)",
}
# default seed of each workload's draws
_SEEDS = {"decode_tiny": 1001, "decode_llama3_8b": 1002, "decode_e4m3_window": 1003, "prefill": 1004,
          "decode_softcap_d256": 1005}


def workload_problem(name: str, seed: int | None = None, batch: int | None = None, **kw) -> Problem:
    """One of the five benchmark workloads (``WORKLOADS``): shapes,
    distributions and options as each is specified.  ``batch`` keeps only the
    first requests (same draws), for reduced cases."""
    if name not in WORKLOADS:
        raise ValueError(f"unknown workload {name!r}")
    seed = _SEEDS[name] if seed is None else seed
    rng = np.random.default_rng(seed + 7919)
    desc = WORKLOADS[name]
    cut = slice(None) if batch is None else slice(0, batch)
    if name == "decode_tiny":
        B = 4
        sl = rng.integers(1, 301, size=B)[cut]
        args = dict(num_q_heads=8, num_kv_heads=2, head_dim=64, page_size=16,
                    seq_lens=sl, scale=64 ** -0.5, pool_pages=128)
        return build_problem("decode", seed=seed, name=desc, **{**args, **kw})
    if name == "decode_llama3_8b":
        B = 64
        sl = rng.integers(512, 8193, size=B)[cut]
        args = dict(num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                    seq_lens=sl, scale=128 ** -0.5)
        return build_problem("decode", seed=seed, name=desc, **{**args, **kw})
    if name == "decode_e4m3_window":
        B = 128
        sl = np.floor(np.exp(rng.uniform(math.log(1024), math.log(32768), size=B))).astype(np.int64)[cut]
        args = dict(num_q_heads=64, num_kv_heads=8, head_dim=64, page_size=64,
                    seq_lens=sl, kv_dtype="fp8_e4m3", k_scale=0.05, v_scale=0.05,
                    window=1024, sinks=True, scale=64 ** -0.5)
        return build_problem("decode", seed=seed, name=desc, **{**args, **kw})
    if name == "prefill":
        B = 8
        ctx = rng.integers(0, 4097, size=B)[cut]
        ql = rng.integers(1, 2049, size=B)[cut]
        args = dict(num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                    seq_lens=ctx + ql, query_lens=ql, scale=128 ** -0.5)
        return build_problem("extend", seed=seed, name=desc, **{**args, **kw})
    B = 256   # decode_softcap_d256
    sl = np.clip(np.rint(rng.lognormal(math.log(2048), 1.0, size=B)), 1, 65536).astype(np.int64)[cut]
    args = dict(num_q_heads=16, num_kv_heads=8, head_dim=256, page_size=32,
                seq_lens=sl, soft_cap=50.0, window=4096, scale=256 ** -0.5)
    return build_problem("decode", seed=seed, name=desc, **{**args, **kw})
