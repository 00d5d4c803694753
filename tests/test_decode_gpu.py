"""Decode parity: the CUDA split-KV path (through the C ABI) against the oracle."""
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


def _small(seed, *, Hq, Hkv, D, ps, lens, kv="bf16", **kw):
    extra = {}
    if kv == "fp8_e4m3":
        extra = dict(k_scale=0.05, v_scale=0.05)
    return wl.build_problem("decode", num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=ps,
                            seq_lens=lens, kv_dtype=kv, seed=seed, **extra, **kw)


LENS = [1, 15, 16, 17, 63, 200, 777, 1500]

VARIANTS = [
    # Hq, Hkv, D, ps, kv
    (8, 2, 64, 16, "bf16"),
    (32, 8, 128, 16, "bf16"),
    (16, 8, 256, 32, "bf16"),
    (64, 8, 64, 64, "fp8_e4m3"),
    (16, 4, 128, 32, "fp8_e4m3"),
    (4, 2, 256, 16, "fp8_e4m3"),
    (16, 1, 128, 16, "bf16"),       # group 16: two 8-head MMA columns
    (12, 1, 64, 32, "bf16"),        # group 12: padded heads
    (4, 4, 128, 64, "bf16"),        # group 1 (MHA)
    (64, 2, 128, 16, "bf16"),       # group 32: two 16-head CTAs per kv head
    (40, 2, 64, 32, "fp8_e4m3"),    # group 20: 16 + 4 heads
]


@pytest.mark.parametrize("Hq,Hkv,D,ps,kv", VARIANTS)
@pytest.mark.parametrize("opts", [{}, {"window": 70, "sinks": True}, {"soft_cap": 5.0, "window": 300}])
def test_decode_variants(Hq, Hkv, D, ps, kv, opts):
    p = _small(Hq * 7 + D + ps, Hq=Hq, Hkv=Hkv, D=D, ps=ps, lens=LENS, kv=kv, **opts)
    ref_o, ref_l = oracle.attention(p)
    for ns in (0, 1, 3):
        out, lse = gh.run(p, num_splits=ns)
        gh.assert_parity(out, lse, ref_o, ref_l, what=f"splits={ns}")


def test_tiny_decode_split_counts():
    p = wl.workload_problem("decode_tiny")
    ref_o, ref_l = oracle.attention(p)
    for ns in (4, 1, 2, 3, 7, 0):
        out, lse = gh.run(p, num_splits=ns)
        gh.assert_parity(out, lse, ref_o, ref_l, what=f"tiny decode, splits={ns}")


def test_split_invariance_close():
    # Different split counts give the same answer up to fp32 re-association.
    p = _small(5, Hq=32, Hkv=8, D=128, ps=16, lens=[5000, 3000, 129])
    outs = [gh.run(p, num_splits=ns) for ns in (1, 2, 5, 16, 0)]
    for o, l in outs[1:]:
        assert np.abs(o - outs[0][0]).max() <= 1e-2
        assert np.abs(l - outs[0][1]).max() <= 1e-4


def test_identity_probe_window_one_bitwise():
    # window = 1: each query sees only its own key -> out == V row exactly,
    # with NaN in every unattended slot of the pool.
    for (Hq, Hkv, D, ps, kv) in VARIANTS:
        p = _small(11 + D, Hq=Hq, Hkv=Hkv, D=D, ps=ps, lens=LENS, kv=kv, window=1, keep_logical=True)
        out, _ = gh.run(p)
        ref_o, _ = oracle.attention(p)
        assert np.array_equal(out.astype(np.float64), ref_o), (Hq, Hkv, D, ps, kv)


def test_onehot_query_reads_exact_key():
    # q = e_d (head h probes dim d = (7h) mod D), scale 1, window 1: the LSE is
    # the dequantised K element at the query's own position.  The kernel's
    # softmax runs in the log2 domain, so LSE = (s*log2 e)*ln 2 may differ from
    # s by a few fp32 ulps; any wrong element differs by >= a bf16 ulp (2^-8).
    for kv in ("bf16", "fp8_e4m3"):
        Hq, Hkv, D, ps = 16, 2, 128, 16
        T = len(LENS)
        qv = np.zeros((T, Hq, D), np.float32)
        dims = [(7 * h) % D for h in range(Hq)]
        for h in range(Hq):
            qv[:, h, dims[h]] = 1.0
        p = _small(21, Hq=Hq, Hkv=Hkv, D=D, ps=ps, lens=LENS, kv=kv, window=1, q_values=qv)
        p.scale = 1.0
        _, lse = gh.run(p)
        _, ref_l = oracle.attention(p)
        err = np.abs(lse.astype(np.float64) - ref_l)
        assert np.all(err <= 4 * np.spacing(np.abs(ref_l).astype(np.float32))), (kv, err.max())


def test_page_permutation_bitwise():
    p = _small(31, Hq=32, Hkv=8, D=128, ps=16, lens=LENS, window=500, sinks=True)
    o1, l1 = gh.run(p)
    rng = np.random.default_rng(3)
    perm = rng.permutation(p.num_pages)
    k2 = np.empty_like(p.k_cache)
    v2 = np.empty_like(p.v_cache)
    k2[perm] = p.k_cache
    v2[perm] = p.v_cache
    bt = p.block_table.copy()
    used = bt != wl.BT_SENTINEL
    bt[used] = perm[bt[used]]
    q = dataclasses.replace(p, k_cache=k2, v_cache=v2, block_table=bt)
    o2, l2 = gh.run(q)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_interleaved_layout_bitwise():
    a = _small(41, Hq=16, Hkv=8, D=256, ps=32, lens=LENS, layout="separate")
    b = _small(41, Hq=16, Hkv=8, D=256, ps=32, lens=LENS, layout="interleaved")
    oa, la = gh.run(a)
    ob, lb = gh.run(b)
    assert np.array_equal(oa, ob) and np.array_equal(la, lb)


def test_empty_and_zero_length():
    p = _small(51, Hq=8, Hkv=2, D=64, ps=16, lens=[0, 5, 0, 40], sinks=True)
    ref_o, ref_l = oracle.attention(p)
    out, lse = gh.run(p)
    gh.assert_parity(out, lse, ref_o, ref_l)
    p.sinks = None
    ref_o, ref_l = oracle.attention(p)
    out, lse = gh.run(p)
    gh.assert_parity(out, lse, ref_o, ref_l)


def test_no_lse_output():
    p = _small(61, Hq=8, Hkv=2, D=64, ps=16, lens=LENS)
    ref_o, _ = oracle.attention(p)
    out, _ = gh.run(p, with_lse=False)
    gh.assert_parity(out, None, ref_o, None)


@pytest.mark.parametrize("name", ["decode_llama3_8b", "decode_e4m3_window", "decode_softcap_d256"])
def test_full_size_decode_workloads_all_rows(name):
    # The benchmark workloads at full size, in the launch configuration the
    # benchmark uses (planner with host lengths); every output element and
    # every LSE of every request and head is compared with the oracle.
    p = wl.workload_problem(name)
    out, lse = gh.run(p)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    ref_o, ref_l = oracle.attention(p)
    eo, el = gh.assert_parity(out, lse, ref_o, ref_l, what=wl.WORKLOADS[name])
    print(f"{name}: all {out.shape[0] * out.shape[1]} rows, max |out err| {eo:.3e}, max |lse err| {el:.3e}")


def test_merge_paths_reuse_one_scratch():
    # Several splits per request.  With a counter per (request, kv head) in the
    # scratch header the split that finishes last merges (one launch); a plan
    # whose capacity exceeds the counters launches the merge kernel.  Each
    # plan's scratch serves three different batches in a row without being
    # re-initialised: every call must leave its counters at zero.
    import torch
    from paged_kv_gqa_12_gb300 import binding as pb
    # one plan per path, so the three batches share its window and sinks
    batches = [[900, 3000, 17, 1], [2500, 5, 1200], [4000, 4000]]
    probs = [wl.build_problem("decode", num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                              seq_lens=lens, window=700, sinks=True, seed=41 + i, bt_width=256)
             for i, lens in enumerate(batches)]
    refs = [oracle.attention(p) for p in probs]
    for max_batch, fused in ((4, 1), (pb.MERGE_COUNTERS // 8 + 1, 0)):
        plan = gh.make_plan(probs[0], num_splits=5, host_lens=False, max_batch=max_batch)
        assert plan.split_merge == fused and plan.launches == 2 - fused and plan.max_splits == 5
        scratch = pb.alloc_scratch(plan)
        for p, (ref_o, ref_l) in zip(probs, refs):
            d = gh.upload(p)
            out = torch.full(p.q.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
            lse = torch.full(p.q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
            pb.decode(plan, d["q"], d["k"], d["v"], d["bt"], d["sl"], scale=p.scale, out=out, lse=lse,
                      sinks=d["sinks"], scratch=scratch)
            torch.cuda.synchronize()
            assert pb.check(scratch) == 0
            gh.assert_parity(out.float().cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l,
                             what=f"max_batch={max_batch}, lens={p.seq_lens.tolist()}")
        # the header's counters are back at zero after the last call
        hdr = scratch[:pb.SCRATCH_HEADER_BYTES].cpu().numpy()
        assert not hdr.any()


def test_length_beyond_capacity_is_flagged_and_scratch_recovers():
    # A request longer than the plan's capacity (block-table width x page
    # size) is refused on the device before anything of it is read; the
    # other requests of the call, split and merged by their last split, are
    # still exact.  After pa_check the same scratch serves the next call.
    import torch
    from paged_kv_gqa_12_gb300 import binding as pb
    W = 16                                                   # 256 keys per request at most
    good = wl.build_problem("decode", num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                            seq_lens=[200, 250, 100], seed=91, bt_width=W)
    plan = gh.make_plan(good)
    assert plan.max_splits > 1 and plan.split_merge == 1
    scratch = pb.alloc_scratch(plan)
    d = gh.upload(good)
    ref_o, ref_l = oracle.attention(good)
    bad_lens = torch.tensor([200, 600, 100], dtype=torch.int32, device="cuda")
    out = torch.full(good.q.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full(good.q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
    pb.decode(plan, d["q"], d["k"], d["v"], d["bt"], bad_lens, scale=good.scale, out=out, lse=lse, scratch=scratch)
    assert pb.check(scratch) == 4                            # length beyond the plan's capacity
    o, l = out.float().cpu().numpy(), lse.cpu().numpy()
    for b in (0, 2):
        gh.assert_parity(o[b:b + 1], l[b:b + 1], ref_o[b:b + 1], ref_l[b:b + 1], what=f"request {b} beside the bad one")
    assert not scratch[:pb.SCRATCH_HEADER_BYTES].cpu().numpy().any()
    out.fill_(float("nan"))
    pb.decode(plan, d["q"], d["k"], d["v"], d["bt"], d["sl"], scale=good.scale, out=out, lse=lse, scratch=scratch)
    assert pb.check(scratch) == 0
    gh.assert_parity(out.float().cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l, what="after recovery")
