"""Per-request e4m3 descales (one k and one v scale per request, fp32 on the
device): decode, verify and extend (both ways an e4m3 cache reaches the
extend kernel) against the oracle, and the per-tensor case bit for bit."""
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


def _scales(seed, B):
    rng = np.random.default_rng(seed)
    # a spread of scales, so one taken from the wrong request shows
    return (np.exp(rng.uniform(np.log(0.01), np.log(0.3), size=B)).astype(np.float32),
            np.exp(rng.uniform(np.log(0.01), np.log(0.3), size=B)).astype(np.float32))


@pytest.mark.parametrize("Hq,Hkv,D,ps", [(64, 8, 64, 64), (16, 4, 128, 32), (40, 2, 64, 32)])
@pytest.mark.parametrize("opts", [{}, {"window": 70, "sinks": True}])
def test_decode_per_request_scales(Hq, Hkv, D, ps, opts):
    lens = [1, 17, 200, 777, 1500, 64]
    ks, vs = _scales(Hq + D, len(lens))
    p = wl.build_problem("decode", num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=ps, seq_lens=lens,
                         kv_dtype="fp8_e4m3", k_scales=ks, v_scales=vs, seed=Hq * 3 + D, **opts)
    ref_o, ref_l = oracle.attention(p)
    for ns in (0, 1, 3):
        out, lse = gh.run(p, num_splits=ns)
        gh.assert_parity(out, lse, ref_o, ref_l, what=f"decode per-request scales, splits={ns}")


def test_verify_per_request_scales():
    ctx = np.array([0, 15, 700, 2047])
    ql = np.full_like(ctx, 2)
    ks, vs = _scales(5, len(ctx))
    p = wl.build_problem("extend", num_q_heads=64, num_kv_heads=8, head_dim=64, page_size=64,
                         seq_lens=ctx + ql, query_lens=ql, kv_dtype="fp8_e4m3", k_scales=ks, v_scales=vs, seed=55,
                         window=300, sinks=True)
    ref_o, ref_l = oracle.attention(p)
    out, lse = gh.run(p, verify=True)
    gh.assert_parity(out, lse, ref_o, ref_l, what="verify per-request scales")


@pytest.mark.parametrize("D", [64, 128, 256])
def test_extend_per_request_scales_both_paths(D):
    from paged_kv_gqa_12_gb300 import binding as pb
    ctx = np.array([0, 5, 300, 1000, 129])
    ql = np.array([37, 1, 200, 64, 300])
    ks, vs = _scales(D, len(ctx))
    p = wl.build_problem("extend", num_q_heads=32, num_kv_heads=8, head_dim=D, page_size=16, seq_lens=ctx + ql,
                         query_lens=ql, kv_dtype="fp8_e4m3", k_scales=ks, v_scales=vs, seed=D + 1)
    ref_o, ref_l = oracle.attention(p)
    d = gh.upload(p)
    copy_plan = gh.make_plan(p)
    tile_plan = pb.plan(mode=pb.MODE_EXTEND, num_q_heads=32, num_kv_heads=8, head_dim=D, page_size=16,
                        kv_dtype=pb.KV_FP8_E4M3, max_batch=p.batch, max_pages_per_seq=1 << 16,
                        max_total_q=p.num_rows)
    assert copy_plan.kv_copy == 1 and tile_plan.kv_copy == 0
    o1, l1 = gh.run(p, d=d, plan=copy_plan)
    gh.assert_parity(o1, l1, ref_o, ref_l, what="extend per-request scales (bf16 copy)")
    o2, l2 = gh.run(p, d=d, plan=tile_plan)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_equal_per_request_scales_are_the_per_tensor_case():
    # the same scale for every request gives the per-tensor result bit for bit
    lens = [1, 17, 200, 777]
    p = wl.build_problem("decode", num_q_heads=64, num_kv_heads=8, head_dim=64, page_size=64, seq_lens=lens,
                         kv_dtype="fp8_e4m3", k_scale=0.05, v_scale=0.07, seed=9)
    o1, l1 = gh.run(p)
    per = dataclasses.replace(p, k_scales=np.full(4, 0.05, np.float32), v_scales=np.full(4, 0.07, np.float32),
                              k_scale=1.0, v_scale=1.0)
    o2, l2 = gh.run(per)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
