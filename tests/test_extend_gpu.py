"""Extend (prefix-prefill) parity: the tcgen05 path (through the C ABI) against the oracle."""
import dataclasses

import numpy as np
import pytest

import oracle
from paged_kv_gqa_12_gb300 import workloads as wl
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_gqa_12_gb300 import binding
    binding.load()


def _ext(seed, *, Hq, Hkv, D, ps, ctx, ql, **kw):
    ctx = np.asarray(ctx)
    ql = np.asarray(ql)
    return wl.build_problem("extend", num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=ps,
                            seq_lens=ctx + ql, query_lens=ql, seed=seed, **kw)


# ragged: empty context, context shorter than a tile, multi-tile context,
# query counts off tile boundaries, a single-query request
CTX = [0, 5, 300, 1000, 129, 0]
QL = [37, 1, 200, 64, 513, 128]

VARIANTS = [
    # Hq, Hkv, D, ps
    (32, 8, 128, 16),
    (8, 2, 64, 16),
    (16, 8, 256, 32),
    (12, 4, 256, 16),     # head_dim 256, group 3: 126 of 128 rows used
    (32, 2, 256, 64),     # head_dim 256, group 16
    (64, 8, 128, 64),     # group 8
    (16, 1, 128, 16),     # group 16
    (8, 8, 64, 32),       # group 1
    (12, 4, 128, 16),     # group 3: 126 of 128 rows used
    (64, 2, 128, 16),     # group 32: 4 tokens per query tile
    (128, 1, 64, 32),     # group 128: one token per query tile
]


@pytest.mark.parametrize("Hq,Hkv,D,ps", VARIANTS)
@pytest.mark.parametrize("opts", [{}, {"window": 100, "sinks": True}, {"soft_cap": 8.0}])
def test_extend_variants(Hq, Hkv, D, ps, opts):
    p = _ext(Hq * 5 + D + ps, Hq=Hq, Hkv=Hkv, D=D, ps=ps, ctx=CTX, ql=QL, **opts)
    ref_o, ref_l = oracle.attention(p)
    out, lse = gh.run(p)
    gh.assert_parity(out, lse, ref_o, ref_l, what=f"extend {Hq},{Hkv},{D},{ps} {opts}")


def test_extend_identity_probe_bitwise():
    # window 1: every query sees only its own key, whose V row must come back
    # exactly; every unattended slot of the pool is NaN.
    for (Hq, Hkv, D, ps) in VARIANTS:
        p = _ext(7 + D, Hq=Hq, Hkv=Hkv, D=D, ps=ps, ctx=CTX, ql=QL, window=1)
        out, _ = gh.run(p)
        ref_o, _ = oracle.attention(p)
        assert np.array_equal(out.astype(np.float64), ref_o), (Hq, Hkv, D, ps)


def test_extend_page_permutation_bitwise():
    p = _ext(17, Hq=32, Hkv=8, D=128, ps=16, ctx=CTX, ql=QL, sinks=True)
    o1, l1 = gh.run(p)
    rng = np.random.default_rng(5)
    perm = rng.permutation(p.num_pages)
    k2 = np.empty_like(p.k_cache)
    v2 = np.empty_like(p.v_cache)
    k2[perm] = p.k_cache
    v2[perm] = p.v_cache
    bt = p.block_table.copy()
    used = bt != wl.BT_SENTINEL
    bt[used] = perm[bt[used]]
    o2, l2 = gh.run(dataclasses.replace(p, k_cache=k2, v_cache=v2, block_table=bt))
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_extend_single_query_matches_decode():
    ctx = np.array([0, 17, 999, 4000])
    e = _ext(27, Hq=32, Hkv=8, D=128, ps=16, ctx=ctx, ql=[1, 1, 1, 1], window=700, sinks=True)
    oe, le = gh.run(e)
    d = dataclasses.replace(e, mode="decode", query_start_loc=None)
    od, ld = gh.run(d)
    ref_o, ref_l = oracle.attention(e)
    gh.assert_parity(oe, le, ref_o, ref_l, what="extend q=1")
    gh.assert_parity(od, ld, ref_o, ref_l, what="decode")


def test_extend_empty_request_rows():
    # zero new tokens for some requests: nothing to compute for them
    p = _ext(37, Hq=8, Hkv=2, D=64, ps=16, ctx=[10, 50, 0, 7], ql=[0, 33, 5, 0])
    ref_o, ref_l = oracle.attention(p)
    out, lse = gh.run(p)
    gh.assert_parity(out, lse, ref_o, ref_l)


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
def test_extend_full_size_workload_all_rows(kv):
    # The extend workload at full size in the benchmark's launch
    # configuration (bf16 cache; e4m3 cache with scales 0.05 through the
    # dequantised bf16 copy the plan chooses): every row of every request,
    # every head, against the oracle.
    extra = dict(kv_dtype="fp8_e4m3", k_scale=0.05, v_scale=0.05) if kv == "fp8_e4m3" else {}
    p = wl.workload_problem("prefill", **extra)
    if kv == "fp8_e4m3":
        assert gh.make_plan(p).kv_copy == 1
    out, lse = gh.run(p)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    ref_o, ref_l = oracle.attention(p)
    eo, el = gh.assert_parity(out, lse, ref_o, ref_l, what=f"extend workload, full size, {kv} cache")
    print(f"extend {kv}: all {p.num_rows} rows x {p.num_q_heads} heads, max |out err| {eo:.3e}, "
          f"max |lse err| {el:.3e}")


FP8_VARIANTS = [(32, 8, 128, 16), (8, 2, 64, 16), (16, 8, 256, 32), (64, 8, 64, 64)]


@pytest.mark.parametrize("Hq,Hkv,D,ps", FP8_VARIANTS)
@pytest.mark.parametrize("opts", [{}, {"window": 100, "sinks": True}, {"soft_cap": 8.0}])
def test_extend_fp8_cache(Hq, Hkv, D, ps, opts):
    # e4m3 cache, dequantised bf16(float(code) * scale) on both sides
    p = _ext(Hq * 3 + D + ps, Hq=Hq, Hkv=Hkv, D=D, ps=ps, ctx=CTX, ql=QL, kv_dtype="fp8_e4m3",
             k_scale=0.05, v_scale=0.07, **opts)
    ref_o, ref_l = oracle.attention(p)
    out, lse = gh.run(p)
    gh.assert_parity(out, lse, ref_o, ref_l, what=f"extend fp8 {Hq},{Hkv},{D},{ps} {opts}")


def test_extend_fp8_identity_probe_bitwise():
    for (Hq, Hkv, D, ps) in FP8_VARIANTS:
        p = _ext(9 + D, Hq=Hq, Hkv=Hkv, D=D, ps=ps, ctx=CTX, ql=QL, kv_dtype="fp8_e4m3", k_scale=0.05,
                 v_scale=0.05, window=1)
        out, _ = gh.run(p)
        ref_o, _ = oracle.attention(p)
        assert np.array_equal(out.astype(np.float64), ref_o), (Hq, Hkv, D, ps)


@pytest.mark.parametrize("D", [64, 128])
def test_extend_fp8_copy_and_in_kernel_paths_agree(D):
    # the e4m3 cache reaches the attention kernel either as a bf16 copy made
    # once per call or dequantised per tile in shared memory: the same bf16
    # values in the same key tiles either way, so the outputs are bitwise
    # equal
    from paged_kv_gqa_12_gb300 import binding as pb
    for opts in ({}, {"window": 100, "sinks": True}):
        p = _ext(71 + D, Hq=32, Hkv=8, D=D, ps=16, ctx=CTX, ql=QL, kv_dtype="fp8_e4m3", k_scale=0.05,
                 v_scale=0.07, **opts)
        d = gh.upload(p)
        copy_plan = gh.make_plan(p)
        assert copy_plan.kv_copy == 1
        tile_plan = pb.plan(mode=pb.MODE_EXTEND, num_q_heads=32, num_kv_heads=8, head_dim=D, page_size=16,
                            kv_dtype=pb.KV_FP8_E4M3, max_batch=p.batch, max_pages_per_seq=1 << 16,
                            max_total_q=p.num_rows, window=p.window, has_sinks=p.sinks is not None)
        assert tile_plan.kv_copy == 0
        o1, l1 = gh.run(p, d=d, plan=copy_plan)
        o2, l2 = gh.run(p, d=d, plan=tile_plan)
        assert copy_plan.tile_tokens == tile_plan.tile_tokens
        assert np.array_equal(o1, o2) and np.array_equal(l1, l2), opts
        ref_o, ref_l = oracle.attention(p)
        gh.assert_parity(o1, l1, ref_o, ref_l, what=f"extend fp8 copy D={D} {opts}")
        gh.assert_parity(o2, l2, ref_o, ref_l, what=f"extend fp8 in-kernel dequantisation D={D} {opts}")


@pytest.mark.parametrize("D", [64, 128, 256])
def test_extend_padded_output_rows(D):
    # output rows 16 elements longer than head_dim: every other (token, head)
    # row starts off a 32-byte boundary, so the epilogue takes its 16-byte
    # stores there and its 32-byte stores elsewhere; the padding stays as set
    import torch
    from paged_kv_gqa_12_gb300 import binding as pb
    p = _ext(211 + D, Hq=16, Hkv=4, D=D, ps=16, ctx=CTX, ql=QL, sinks=True)
    d = gh.upload(p)
    plan = gh.make_plan(p)
    T, Hq = p.q.shape[0], p.q.shape[1]
    full = torch.full((T, Hq, D + 8), 3.0, dtype=torch.bfloat16, device="cuda")
    out = full.narrow(2, 0, D)
    lse = torch.empty((T, Hq), dtype=torch.float32, device="cuda")
    scratch = pb.alloc_scratch(plan)
    pb.extend(plan, d["q"], d["k"], d["v"], d["bt"], d["sl"], d["qsl"], scale=p.scale, out=out, lse=lse,
              sinks=d["sinks"], scratch=scratch)
    assert pb.check(scratch) == 0
    ref_o, ref_l = oracle.attention(p)
    gh.assert_parity(out.float().cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l, what=f"extend padded rows D={D}")
    assert bool((full[:, :, D:] == 3.0).all())


@pytest.mark.parametrize("opts", [{}, {"window": 4096, "sinks": True}])
def test_extend_long_context_sampled(opts):
    # contexts of 20-32K keys: work items of several hundred key tiles; the
    # oracle checks the first and last rows of each request and a sample
    ctx = np.array([32000, 20000, 7])
    ql = np.array([300, 1000, 129])
    p = _ext(91, Hq=32, Hkv=8, D=128, ps=16, ctx=ctx, ql=ql, **opts)
    out, lse = gh.run(p)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    qsl = p.query_start_loc
    rng = np.random.default_rng(6)
    rows = [int(qsl[b]) for b in range(p.batch)] + [int(qsl[b + 1]) - 1 for b in range(p.batch)]
    rows += list(rng.choice(p.num_rows, size=24, replace=False))
    rows = np.unique(np.array(rows, np.int32))
    ref_o, ref_l = oracle.attention(p, rows=rows)
    gh.assert_parity(out[rows], lse[rows], ref_o, ref_l, what=f"extend long context {opts}")
