"""Capacity plans are replayable: pa_decode and pa_extend captured once in a
CUDA graph, then replayed after the device buffers were refilled with a
different batch (other lengths, other pages, other values, same capacities)."""
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


POOL, WIDTH = 900, 80


def _decode(seed, lens):
    return wl.build_problem("decode", num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                            seq_lens=lens, seed=seed, window=900, sinks=True,
                            pool_pages=POOL, bt_width=WIDTH)


def _extend(seed, ctx, ql, **kw):
    ctx, ql = np.asarray(ctx), np.asarray(ql)
    return wl.build_problem("extend", num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                            seq_lens=ctx + ql, query_lens=ql, seed=seed, pool_pages=POOL, bt_width=WIDTH, **kw)


def _fill(dst, p):
    src = gh.upload(p)
    for k in ("q", "k", "v", "bt", "sl", "qsl", "sinks", "k_scales", "v_scales"):
        if dst.get(k) is not None:
            dst[k].copy_(src[k])


def _graph_roundtrip(first, second):
    import torch
    from paged_kv_gqa_12_gb300 import binding as pb
    d = gh.upload(first)
    plan = gh.make_plan(first, host_lens=False, max_batch=first.batch)   # capacities only
    scratch = pb.alloc_scratch(plan)
    out = torch.zeros(first.q.shape, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(first.q.shape[:2], dtype=torch.float32, device="cuda")
    kw = dict(scale=first.scale, out=out, lse=lse, sinks=d["sinks"], scratch=scratch, k_scale=first.k_scale,
              v_scale=first.v_scale, k_scales=d.get("k_scales"), v_scales=d.get("v_scales"))

    def call():
        if first.mode == "decode":
            pb.decode(plan, d["q"], d["k"], d["v"], d["bt"], d["sl"], **kw)
        else:
            pb.extend(plan, d["q"], d["k"], d["v"], d["bt"], d["sl"], d["qsl"], **kw)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()                      # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    results = []
    for p in (first, second):
        _fill(d, p)
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert pb.check(scratch) == 0
        results.append((out.float().cpu().numpy(), lse.cpu().numpy()))
    return results


def test_decode_graph_replay_with_new_batch():
    a = _decode(501, [1200, 5, 700, 1000, 33, 999])
    b = _decode(502, [17, 1279, 640, 1, 900, 1100])
    (oa, la), (ob, lb) = _graph_roundtrip(a, b)
    for p, o, l in ((a, oa, la), (b, ob, lb)):
        ref_o, ref_l = oracle.attention(p)
        gh.assert_parity(o, l, ref_o, ref_l, what="graph replay decode")


def test_extend_graph_replay_with_new_batch():
    a = _extend(511, [100, 0, 700, 1000], [60, 200, 3, 137])
    b = _extend(512, [0, 950, 20, 333], [150, 50, 150, 50])      # same total rows (400)
    (oa, la), (ob, lb) = _graph_roundtrip(a, b)
    for p, o, l in ((a, oa, la), (b, ob, lb)):
        ref_o, ref_l = oracle.attention(p)
        gh.assert_parity(o, l, ref_o, ref_l, what="graph replay extend")


def test_extend_e4m3_graph_replay_with_new_scales():
    # e4m3 cache through the bf16 copy (one more captured kernel), per-request
    # scales read from device memory on every replay
    a = _extend(521, [100, 0, 700, 1000], [60, 200, 3, 137], kv_dtype="fp8_e4m3",
                k_scales=[0.05, 0.1, 0.02, 0.07], v_scales=[0.03, 0.2, 0.05, 0.01])
    b = _extend(522, [0, 950, 20, 333], [150, 50, 150, 50], kv_dtype="fp8_e4m3",
                k_scales=[0.2, 0.01, 0.06, 0.04], v_scales=[0.1, 0.05, 0.3, 0.02])
    (oa, la), (ob, lb) = _graph_roundtrip(a, b)
    for p, o, l in ((a, oa, la), (b, ob, lb)):
        ref_o, ref_l = oracle.attention(p)
        gh.assert_parity(o, l, ref_o, ref_l, what="graph replay extend e4m3")
