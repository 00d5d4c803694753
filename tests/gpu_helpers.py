"""Helpers shared by the GPU parity tests: upload a generated problem, run the
CUDA path through the C ABI, and compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

from paged_kv_gqa_12_gb300 import binding as pb

OUT_ATOL = 1e-2     # bf16 output, max-abs against the fp32/fp64 oracle
LSE_ATOL = 1e-3     # fp32 LSE


def _t(a: np.ndarray) -> torch.Tensor:
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a))


def upload(p, device="cuda"):
    d = {}
    d["q"] = _t(p.q).to(device)
    if p.kv_storage is not None:
        st = _t(p.kv_storage).to(device)
        es = [s // p.k_cache.itemsize for s in p.k_cache.strides]
        d["k"] = torch.as_strided(st, p.k_cache.shape, es, 0)
        d["v"] = torch.as_strided(st, p.v_cache.shape, es, (p.v_cache.ctypes.data - p.kv_storage.ctypes.data) // p.k_cache.itemsize)
        d["storage"] = st
    else:
        d["k"] = _t(p.k_cache).to(device)
        d["v"] = _t(p.v_cache).to(device)
    d["bt"] = torch.from_numpy(p.block_table).to(device)
    d["sl"] = torch.from_numpy(p.seq_lens).to(device)
    d["qsl"] = None if p.query_start_loc is None else torch.from_numpy(p.query_start_loc).to(device)
    d["sinks"] = None if p.sinks is None else torch.from_numpy(p.sinks).to(device)
    ks, vs = getattr(p, "k_scales", None), getattr(p, "v_scales", None)
    d["k_scales"] = None if ks is None else torch.from_numpy(np.ascontiguousarray(ks, np.float32)).to(device)
    d["v_scales"] = None if vs is None else torch.from_numpy(np.ascontiguousarray(vs, np.float32)).to(device)
    return d


def make_plan(p, num_splits=0, host_lens=True, max_batch=None, verify=False):
    kv = pb.KV_FP8_E4M3 if p.kv_dtype == "fp8_e4m3" else pb.KV_BF16
    mode = pb.MODE_DECODE if p.mode == "decode" else pb.MODE_EXTEND
    q_len = 0
    if verify:
        ql = p.query_lens()
        assert p.mode == "extend" and np.all(ql == ql[0]), "verify needs equal query counts"
        mode, q_len = pb.MODE_VERIFY, int(ql[0])
    return pb.plan(mode=mode, num_q_heads=p.num_q_heads, num_kv_heads=p.num_kv_heads,
                   head_dim=p.head_dim, page_size=p.page_size, kv_dtype=kv,
                   max_batch=max_batch or max(p.batch, 1), max_pages_per_seq=p.block_table.shape[1],
                   max_total_q=max(p.num_rows, 1), window=p.window, has_sinks=p.sinks is not None,
                   soft_cap=p.soft_cap, num_splits=num_splits, q_len=q_len,
                   host_seq_lens=p.seq_lens if (host_lens and (p.mode == "decode" or verify)) else None)


def run(p, d=None, plan=None, num_splits=0, host_lens=True, with_lse=True, verify=False):
    """Run decode or extend on the GPU; returns (out float32 [T,Hq,D], lse [T,Hq]) on the host."""
    d = d or upload(p)
    plan = plan or make_plan(p, num_splits=num_splits, host_lens=host_lens, verify=verify)
    T, Hq, D = p.q.shape
    out = torch.full((T, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((T, Hq), float("nan"), dtype=torch.float32, device="cuda") if with_lse else None
    scratch = pb.alloc_scratch(plan)
    kw = dict(scale=p.scale, out=out, lse=lse, sinks=d["sinks"], k_scale=p.k_scale, v_scale=p.v_scale,
              k_scales=d.get("k_scales"), v_scales=d.get("v_scales"), scratch=scratch)
    if p.mode == "decode":
        pb.decode(plan, d["q"], d["k"], d["v"], d["bt"], d["sl"], **kw)
    else:
        pb.extend(plan, d["q"], d["k"], d["v"], d["bt"], d["sl"], d["qsl"], **kw)
    code = pb.check(scratch)
    assert code == 0, f"device error code {code}"
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), (lse.cpu().numpy() if with_lse else None)


def out_tolerance(ref: np.ndarray) -> np.ndarray:
    """1e-2 absolute, widened only where the bf16 output itself cannot be
    closer: half a bf16 ulp of the reference value plus 1e-3."""
    a = np.abs(ref)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    half_ulp = 2.0 ** (e - 8)
    return np.maximum(OUT_ATOL, half_ulp + 1e-3)


def assert_parity(out, lse, ref_out, ref_lse, what=""):
    assert out.shape == ref_out.shape, (out.shape, ref_out.shape)
    assert np.isfinite(out).all(), f"{what}: non-finite outputs"
    err = np.abs(out.astype(np.float64) - ref_out)
    tol = out_tolerance(ref_out)
    bad = err > tol
    assert not bad.any(), (f"{what}: {int(bad.sum())} outputs off; max err {err.max():.3e} "
                           f"at {np.unravel_index(err.argmax(), err.shape)}")
    if lse is not None:
        ninf = np.isneginf(ref_lse)
        assert np.array_equal(np.isneginf(lse), ninf), f"{what}: -inf LSE pattern differs"
        le = np.abs(lse[~ninf].astype(np.float64) - ref_lse[~ninf])
        assert le.size == 0 or le.max() <= LSE_ATOL, f"{what}: LSE max err {le.max():.3e}"
    if lse is None or not np.isfinite(ref_lse).any():
        return float(err.max()), 0.0
    fin = np.isfinite(ref_lse)
    return float(err.max()), float(np.abs(lse[fin].astype(np.float64) - ref_lse[fin]).max())
