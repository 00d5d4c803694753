"""pa_decode_static_scratch: decode for callers that cannot allocate a
workspace (the library's own fixed device array stands in for the caller's
scratch buffer).

Its results must match pa_decode with a caller-provided scratch buffer, on
two calls in a row -- the second call finds the first call's partials still
in the shared array and must not be affected by them.  This file is named so
that pytest collects it last.
"""
import numpy as np
import pytest

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


def _problem(seed, lens, **kw):
    return wl.build_problem("decode", num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                            seq_lens=lens, seed=seed, **kw)


def _run(pb, p, use_static, num_splits):
    import torch
    from tests import gpu_helpers as gh
    d = gh.upload(p)
    plan = gh.make_plan(p, num_splits=num_splits)
    out = torch.full(p.q.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full(p.q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
    kw = dict(scale=p.scale, out=out, lse=lse, sinks=d["sinks"], k_scale=p.k_scale, v_scale=p.v_scale)
    if use_static:
        pb.decode_static_scratch(plan, d["q"], d["k"], d["v"], d["bt"], d["sl"], **kw)
    else:
        scratch = pb.alloc_scratch(plan)
        pb.decode(plan, d["q"], d["k"], d["v"], d["bt"], d["sl"], scratch=scratch, **kw)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy()


def test_static_scratch_matches_caller_scratch_twice(pb):
    from tests import gpu_helpers as gh
    a = _problem(901, [3000, 1, 517, 4096, 77])
    b = _problem(902, [2500, 640, 16, 1999], window=700, sinks=True)
    # two calls in a row through the static workspace, several splits each
    sa = _run(pb, a, True, 4)
    sb = _run(pb, b, True, 3)
    ra = _run(pb, a, False, 4)
    rb = _run(pb, b, False, 3)
    for (so, sl), (ro, rl) in ((sa, ra), (sb, rb)):
        assert np.isfinite(so).all() and np.isfinite(sl).all()
        assert np.abs(so - ro).max() <= gh.OUT_ATOL
        assert np.abs(sl - rl).max() <= gh.LSE_ATOL


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
