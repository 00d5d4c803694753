"""Verify mode (speculative decoding): every request brings the same small
number of new tokens over a long context.  Run through pa_extend with a
verify plan on the split-KV kernels; checked against the oracle's extend."""
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


def _verify(seed, *, Hq, Hkv, D, ps, ctx, q_len, kv="bf16", **kw):
    ctx = np.asarray(ctx)
    ql = np.full_like(ctx, q_len)
    extra = dict(k_scale=0.05, v_scale=0.05) if kv == "fp8_e4m3" else {}
    return wl.build_problem("extend", num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=ps,
                            seq_lens=ctx + ql, query_lens=ql, kv_dtype=kv, seed=seed, **extra, **kw)


CTX = [0, 3, 15, 700, 2047, 5000]

CASES = [
    # Hq, Hkv, D, ps, q_len, kv
    (32, 8, 128, 16, 4, "bf16"),      # Llama-3-8B shape, 3 speculative tokens: 16 rows
    (32, 8, 128, 16, 2, "bf16"),
    (64, 8, 64, 64, 2, "fp8_e4m3"),   # group 8, fp8 cache
    (16, 8, 256, 32, 5, "bf16"),      # group 2, 10 rows
    (16, 1, 128, 16, 1, "bf16"),      # group 16, one token (= decode)
]


@pytest.mark.parametrize("Hq,Hkv,D,ps,q_len,kv", CASES)
@pytest.mark.parametrize("opts", [{}, {"window": 300, "sinks": True}, {"soft_cap": 10.0}])
def test_verify_matches_oracle(Hq, Hkv, D, ps, q_len, kv, opts):
    p = _verify(Hq + D + q_len, Hq=Hq, Hkv=Hkv, D=D, ps=ps, ctx=CTX, q_len=q_len, kv=kv, **opts)
    ref_o, ref_l = oracle.attention(p)
    for ns in (0, 1, 3):
        out, lse = gh.run(p, verify=True, num_splits=ns)
        gh.assert_parity(out, lse, ref_o, ref_l, what=f"verify splits={ns}")


def test_verify_identity_probe_bitwise():
    p = _verify(77, Hq=32, Hkv=8, D=128, ps=16, ctx=CTX, q_len=4, window=1)
    out, _ = gh.run(p, verify=True)
    ref_o, _ = oracle.attention(p)
    assert np.array_equal(out.astype(np.float64), ref_o)


def test_verify_agrees_with_extend_kernel():
    p = _verify(78, Hq=32, Hkv=8, D=128, ps=16, ctx=CTX, q_len=3, sinks=True)
    ov, lv = gh.run(p, verify=True)
    oe, le = gh.run(p)
    assert np.abs(ov - oe).max() <= 2 * gh.OUT_ATOL
    assert np.abs(lv - le).max() <= 2 * gh.LSE_ATOL


def test_verify_rejects_unequal_packing():
    # right row count, wrong packing: the device flags it and leaves the
    # request alone; the host sees the code through pa_check
    import torch
    from paged_kv_gqa_12_gb300 import binding as pb
    p = _verify(79, Hq=32, Hkv=8, D=128, ps=16, ctx=[10, 20], q_len=2)
    plan = gh.make_plan(p, verify=True)
    q2 = wl.build_problem("extend", num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                          seq_lens=[13, 21], query_lens=[3, 1], seed=80)
    d = gh.upload(q2)
    out = torch.zeros(q2.q.shape, dtype=torch.bfloat16, device="cuda")
    scratch = pb.alloc_scratch(plan)
    pb.extend(plan, d["q"], d["k"], d["v"], d["bt"], d["sl"], d["qsl"], scale=q2.scale, out=out,
              scratch=scratch)
    assert pb.check(scratch) != 0
    assert pb.check(scratch) == 0          # pa_check clears the error word
    # the wrong row count is refused on the host
    q3 = wl.build_problem("extend", num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                          seq_lens=[13, 22], query_lens=[3, 2], seed=81)
    d3 = gh.upload(q3)
    out3 = torch.zeros(q3.q.shape, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pb.PaError):
        pb.extend(plan, d3["q"], d3["k"], d3["v"], d3["bt"], d3["sl"], d3["qsl"], scale=q3.scale, out=out3,
                  scratch=scratch)


def test_verify_full_size_all_rows():
    # The benchmark's verify measurement at full size, in its launch
    # configuration: the Llama-3-8B-shaped decode workload's cache and
    # lengths, 4 new query tokens per request (their K/V already in the
    # pages), a verify plan from host lengths; every row against the oracle.
    import dataclasses
    dp = wl.workload_problem("decode_llama3_8b")
    q_len = 4
    rng = np.random.default_rng(77)
    q = wl._to_bf16_bits(rng.standard_normal((dp.batch * q_len, dp.num_q_heads, dp.head_dim), dtype=np.float32))
    p = dataclasses.replace(dp, mode="extend", q=q,
                            query_start_loc=np.arange(0, dp.batch * q_len + 1, q_len, dtype=np.int32))
    out, lse = gh.run(p, verify=True)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    ref_o, ref_l = oracle.attention(p)
    eo, el = gh.assert_parity(out, lse, ref_o, ref_l, what="verify, decode workload, full size")
    print(f"verify q_len 4: all {p.num_rows} rows, max |out err| {eo:.3e}, max |lse err| {el:.3e}")
