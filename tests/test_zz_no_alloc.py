"""pa_decode_static_scratch: decode for callers that cannot allocate a
workspace -- a plugin or host runtime with no device allocator of its own, a
process whose memory pool already owns the whole GPU, or code that must never
allocate so that its latency stays fixed.  The library's own fixed device
array stands in for the caller's scratch buffer.

The entry point runs the same kernels with the same plan as pa_decode, so on
the same inputs its outputs and LSEs must be bitwise equal to pa_decode's with
a caller-provided scratch buffer; both must also match the oracle.  Three
calls run in a row through the static array -- each finds the previous call's
partials and counters in the shared array and must not be affected by them --
covering both merge paths: the last split of each (request, kv head) merging
in the split kernel, and a plan whose (request, kv head) pairs exceed the
header's arrival counters, so a merge kernel follows.  This file is named so
that pytest collects it last.
"""
import numpy as np
import pytest

import oracle
from paged_kv_gqa_12_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pb():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_gqa_12_gb300 import binding
    binding.load()
    return binding


def _cases(pb):
    from tests import gpu_helpers as gh
    a = wl.build_problem("decode", num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                         seq_lens=[3000, 1, 517, 4096, 77], seed=901)
    b = wl.build_problem("decode", num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                         seq_lens=[2500, 640, 16, 1999], seed=902, window=700, sinks=True)
    # more (request, kv head) pairs in the plan's capacity than the scratch
    # header has arrival counters: a separate merge kernel; its partials
    # (2041 requests x 8 heads x 2 splits x 64 dims, fp32) fit in 16 MiB
    c = wl.build_problem("decode", num_q_heads=8, num_kv_heads=8, head_dim=64, page_size=16,
                         seq_lens=[1500, 33, 900], seed=903, sinks=True)
    pa = gh.make_plan(a, num_splits=4)
    pb_ = gh.make_plan(b, num_splits=3)
    pc = gh.make_plan(c, num_splits=2, host_lens=False, max_batch=pb.MERGE_COUNTERS // 8 + 1)
    assert pa.split_merge == 1 and pb_.split_merge == 1
    assert pc.split_merge == 0 and pc.launches == 2 and pc.scratch_bytes <= (16 << 20)
    return [(a, pa), (b, pb_), (c, pc)]


def _run(pb, p, plan, use_static):
    import torch
    from tests import gpu_helpers as gh
    d = gh.upload(p)
    out = torch.full(p.q.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full(p.q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
    kw = dict(scale=p.scale, out=out, lse=lse, sinks=d["sinks"], k_scale=p.k_scale, v_scale=p.v_scale)
    if use_static:
        pb.decode_static_scratch(plan, d["q"], d["k"], d["v"], d["bt"], d["sl"], **kw)
    else:
        scratch = pb.alloc_scratch(plan)
        pb.decode(plan, d["q"], d["k"], d["v"], d["bt"], d["sl"], scratch=scratch, **kw)
        assert pb.check(scratch) == 0
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy()


def test_static_scratch_equals_caller_scratch_and_oracle(pb):
    from tests import gpu_helpers as gh
    cases = _cases(pb)
    # three calls in a row through the static workspace, then the same three
    # through pa_decode with caller-owned scratch buffers
    static = [_run(pb, p, plan, True) for p, plan in cases]
    caller = [_run(pb, p, plan, False) for p, plan in cases]
    for (p, plan), (so, sl), (ro, rl) in zip(cases, static, caller):
        assert np.isfinite(so).all() and np.isfinite(sl).all()
        assert np.array_equal(so, ro) and np.array_equal(sl, rl), f"split_merge={plan.split_merge}"
        ref_o, ref_l = oracle.attention(p)
        gh.assert_parity(so, sl, ref_o, ref_l, what=f"static scratch, split_merge={plan.split_merge}")


def test_static_scratch_rejects_oversized_plan(pb):
    # 256 requests x 64 heads x 64 splits x 256 dims of fp32 partials >> 16 MiB
    plan = pb.plan(mode=pb.MODE_DECODE, num_q_heads=64, num_kv_heads=8, head_dim=256, page_size=16,
                   max_batch=256, max_pages_per_seq=4096, num_splits=64)
    assert plan.scratch_bytes > (16 << 20)
    import torch
    q = torch.zeros((1, 64, 256), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((1, 16, 8, 256), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    sl = torch.ones((1,), dtype=torch.int32, device="cuda")
    out = torch.zeros_like(q)
    with pytest.raises(pb.PaError) as ei:
        pb.decode_static_scratch(plan, q, kv, kv, bt, sl, scale=0.0625, out=out)
    assert ei.value.status == pb.PA_ERR_SCRATCH_TOO_SMALL
