"""KV append (the cache write side): pa_append_kv against the oracle's append,
byte for byte, and an append -> extend round trip against the oracle."""
import dataclasses

import numpy as np
import pytest

import oracle
from paged_kv_gqa_12_gb300 import workloads as wl
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pb():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_gqa_12_gb300 import binding
    binding.load()
    return binding


def _new_tokens(seed, T, Hkv, D, spread=1.0):
    # N(0,1) like every workload (the attention tolerance is stated for it);
    # the byte-exact append tests widen the spread to reach saturation
    rng = np.random.default_rng(seed)
    k = wl._to_bf16_bits(rng.standard_normal((T, Hkv, D), dtype=np.float32) * spread)
    v = wl._to_bf16_bits(rng.standard_normal((T, Hkv, D), dtype=np.float32) * spread)
    return k, v


@pytest.mark.parametrize("kv,layout,D", [("bf16", "separate", 128), ("fp8_e4m3", "separate", 128),
                                         ("fp8_e4m3", "interleaved", 64), ("bf16", "interleaved", 256),
                                         ("fp8_e4m3", "separate", 256)])
def test_append_matches_oracle_bytes(pb, kv, layout, D):
    import torch
    extra = dict(k_scale=0.05, v_scale=0.07) if kv == "fp8_e4m3" else {}
    base = wl.build_problem("decode", num_q_heads=16, num_kv_heads=4, head_dim=D, page_size=16,
                            seq_lens=[100, 37, 250], kv_dtype=kv, layout=layout, seed=301, **extra)
    T = 200
    k_new, v_new = _new_tokens(302, T, 4, D, spread=30.0)   # reaches e4m3 saturation at scale 0.05
    rng = np.random.default_rng(303)
    slots = rng.choice(base.num_pages * 16, size=T, replace=False).astype(np.int64)
    slots[::17] = -1                                          # padding tokens
    # oracle on a host copy
    href = dataclasses.replace(base, kv_storage=None, k_cache=base.k_cache.copy(), v_cache=base.v_cache.copy())
    oracle.append_kv(k_new, v_new, href.k_cache, href.v_cache, slots, base.k_scale, base.v_scale)
    # GPU
    d = gh.upload(base)
    kt = torch.from_numpy(k_new.view(np.int16)).view(torch.bfloat16).cuda()
    vt = torch.from_numpy(v_new.view(np.int16)).view(torch.bfloat16).cuda()
    st = torch.from_numpy(slots).cuda()
    kvd = pb.KV_FP8_E4M3 if kv == "fp8_e4m3" else pb.KV_BF16
    pb.append_kv(kt, vt, d["k"], d["v"], st, kv_dtype=kvd, k_scale=base.k_scale, v_scale=base.v_scale)
    torch.cuda.synchronize()
    got_k = d["k"].cpu().numpy() if kv == "fp8_e4m3" else d["k"].cpu().view(torch.int16).numpy().view(np.uint16)
    got_v = d["v"].cpu().numpy() if kv == "fp8_e4m3" else d["v"].cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got_k, href.k_cache)
    assert np.array_equal(got_v, href.v_cache)


def test_append_reports_slot_outside_pool(pb):
    import torch
    base = wl.build_problem("decode", num_q_heads=8, num_kv_heads=2, head_dim=64, page_size=16,
                            seq_lens=[20], seed=311)
    k_new, v_new = _new_tokens(312, 3, 2, 64)
    slots = np.array([0, base.num_pages * 16 + 5, 17], np.int64)
    d = gh.upload(base)
    kt = torch.from_numpy(k_new.view(np.int16)).view(torch.bfloat16).cuda()
    vt = torch.from_numpy(v_new.view(np.int16)).view(torch.bfloat16).cuda()
    plan = gh.make_plan(base)
    scratch = pb.alloc_scratch(plan)
    pb.append_kv(kt, vt, d["k"], d["v"], torch.from_numpy(slots).cuda(), scratch=scratch)
    assert pb.check(scratch) == pb.DEVICE_PAGE_ID
    k = d["k"].cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(k[0, 0], k_new[0]) and np.array_equal(k[1, 1], k_new[2])


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
def test_append_then_extend(pb, kv):
    # prefill step as the backend runs it: append the new tokens' K/V, then
    # attend from the new queries over the cached context and themselves
    import torch
    extra = dict(k_scale=0.05, v_scale=0.05) if kv == "fp8_e4m3" else {}
    ctx = np.array([300, 0, 1000])
    ql = np.array([100, 70, 3])
    p = wl.build_problem("extend", num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                         seq_lens=ctx + ql, query_lens=ql, kv_dtype=kv, seed=321, **extra)
    # the new tokens' K/V, and where they go
    T = int(ql.sum())
    k_new, v_new = _new_tokens(322, T, 8, 128)
    slots = []
    for b in range(p.batch):
        for i in range(int(ql[b])):
            pos = int(ctx[b]) + i
            slots.append(int(p.block_table[b, pos // 16]) * 16 + pos % 16)
    slots = np.array(slots, np.int64)
    # expected cache and attention from the oracle
    q_ref = dataclasses.replace(p, k_cache=p.k_cache.copy(), v_cache=p.v_cache.copy(), kv_storage=None)
    oracle.append_kv(k_new, v_new, q_ref.k_cache, q_ref.v_cache, slots, p.k_scale, p.v_scale)
    ref_o, ref_l = oracle.attention(q_ref)
    # GPU: append into the device cache, then extend
    d = gh.upload(p)
    kvd = pb.KV_FP8_E4M3 if kv == "fp8_e4m3" else pb.KV_BF16
    pb.append_kv(torch.from_numpy(k_new.view(np.int16)).view(torch.bfloat16).cuda(),
                 torch.from_numpy(v_new.view(np.int16)).view(torch.bfloat16).cuda(), d["k"], d["v"],
                 torch.from_numpy(slots).cuda(), kv_dtype=kvd, k_scale=p.k_scale, v_scale=p.v_scale)
    out, lse = gh.run(p, d=d)
    gh.assert_parity(out, lse, ref_o, ref_l, what=f"append+extend {kv}")
