"""Block-table entries outside the page pool.

The block table maps token j of request b to page block_table[b][j / ps]
("vllm/attention/ops/triton_decode_attention.py", _fwd_grouped_kernel_stage1:
Req_to_tokens addressing).  An entry outside [0, num_pages) for a page that
holds attended keys is a caller error: the kernels read that page as zeros
(an out-of-range TMA box), set PA_DEVICE_PAGE_ID in the scratch error word
and leave every other page and request alone.  The oracle refuses such
entries outright, so the other requests' rows are compared with the oracle
evaluated on those rows only.
"""
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


def _corrupt(p, entries):
    """Block table with (request, page index, value) entries overwritten."""
    bt = p.block_table.copy()
    for b, i, v in entries:
        bt[b, i] = v
    return bt


def _run_flagged(pb, p, bt, plan):
    import torch
    d = gh.upload(p)
    d["bt"] = torch.from_numpy(bt).cuda()
    T, Hq, D = p.q.shape
    out = torch.full((T, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((T, Hq), float("nan"), dtype=torch.float32, device="cuda")
    scratch = pb.alloc_scratch(plan)
    kw = dict(scale=p.scale, out=out, lse=lse, sinks=d["sinks"], k_scale=p.k_scale, v_scale=p.v_scale,
              scratch=scratch)
    if p.mode == "decode":
        pb.decode(plan, d["q"], d["k"], d["v"], d["bt"], d["sl"], **kw)
    else:
        pb.extend(plan, d["q"], d["k"], d["v"], d["bt"], d["sl"], d["qsl"], **kw)
    code = pb.check(scratch)
    assert pb.check(scratch) == 0            # pa_check cleared the header
    return code, out.float().cpu().numpy(), lse.cpu().numpy()


def _rows_of(p, reqs):
    if p.mode == "decode":
        return np.array(reqs, np.int32)
    qsl = p.query_start_loc
    return np.concatenate([np.arange(qsl[b], qsl[b + 1]) for b in reqs]).astype(np.int32)


def _check_others(p, out, lse, good):
    rows = _rows_of(p, good)
    ref_o, ref_l = oracle.attention(p, rows=rows)
    gh.assert_parity(out[rows], lse[rows], ref_o, ref_l, what="requests beside the bad entries")


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
def test_decode_flags_out_of_pool_pages(pb, kv):
    extra = dict(k_scale=0.05, v_scale=0.05) if kv == "fp8_e4m3" else {}
    p = wl.build_problem("decode", num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                         seq_lens=[900, 3000, 17, 1200, 40], seed=501, kv_dtype=kv, window=700, sinks=True,
                         **extra)
    # request 1: a page inside its window; request 3: its last page
    bt = _corrupt(p, [(1, 2500 // 16, p.num_pages + 3), (3, 1199 // 16, -1)])
    for ns in (0, 1, 4):
        code, out, lse = _run_flagged(pb, p, bt, gh.make_plan(p, num_splits=ns))
        assert code == pb.DEVICE_PAGE_ID, (ns, code)
        assert np.isfinite(out).all()
        _check_others(p, out, lse, [0, 2, 4])


@pytest.mark.parametrize("kv,D", [("bf16", 128), ("fp8_e4m3", 64)])
def test_decode_ignores_entries_before_the_window(pb, kv, D):
    # pages wholly before the window are never attended: whatever their
    # entries hold, the call is clean and exact.  With the e4m3 head_dim-64
    # kernel a 32-key tile spans two 16-key pages, so the page just before the
    # window start (keys 2496..2511 of request 0; the window keeps 2512..2999)
    # shares the first tile with attended keys: it is fetched, masked, and must
    # not be flagged.
    extra = dict(k_scale=0.05, v_scale=0.05) if kv == "fp8_e4m3" else {}
    Hq = 64 if D == 64 else 32
    p = wl.build_problem("decode", num_q_heads=Hq, num_kv_heads=8, head_dim=D, page_size=16,
                         seq_lens=[3000, 2000], seed=502, window=488, kv_dtype=kv, **extra)
    bt = _corrupt(p, [(0, 2496 // 16, -7), (0, 3, p.num_pages + 1), (1, 0, p.num_pages + 100)])
    code, out, lse = _run_flagged(pb, p, bt, gh.make_plan(p))
    assert code == 0
    ref_o, ref_l = oracle.attention(p)
    gh.assert_parity(out, lse, ref_o, ref_l, what="entries before the window")


def test_verify_flags_out_of_pool_pages(pb):
    ctx = np.array([700, 2047, 5000])
    p = wl.build_problem("extend", num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                         seq_lens=ctx + 4, query_lens=np.full(3, 4), seed=503)
    bt = _corrupt(p, [(1, 100, p.num_pages)])
    code, out, lse = _run_flagged(pb, p, bt, gh.make_plan(p, verify=True))
    assert code == pb.DEVICE_PAGE_ID
    _check_others(p, out, lse, [0, 2])


@pytest.mark.parametrize("kv,copy", [("bf16", None), ("fp8_e4m3", True), ("fp8_e4m3", False)])
def test_extend_flags_out_of_pool_pages(pb, kv, copy):
    extra = dict(k_scale=0.05, v_scale=0.07) if kv == "fp8_e4m3" else {}
    ctx = np.array([300, 1000, 0, 129])
    ql = np.array([200, 64, 513, 37])
    p = wl.build_problem("extend", num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                         seq_lens=ctx + ql, query_lens=ql, seed=504, kv_dtype=kv, **extra)
    # request 1: a context page; request 2: a page of its new tokens
    bt = _corrupt(p, [(1, 10, p.num_pages + 3), (2, 20, -1)])
    plan = gh.make_plan(p)
    if copy is False:
        plan = pb.plan(mode=pb.MODE_EXTEND, num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                       kv_dtype=pb.KV_FP8_E4M3, max_batch=p.batch, max_pages_per_seq=1 << 16,
                       max_total_q=p.num_rows)
    if copy is not None:
        assert plan.kv_copy == (1 if copy else 0)
    code, out, lse = _run_flagged(pb, p, bt, plan)
    assert code == pb.DEVICE_PAGE_ID
    assert np.isfinite(out).all()
    _check_others(p, out, lse, [0, 3])
