"""The benchmark's algorithmic work (the numerators of every reported
roofline fraction), counted here one key at a time from the definition:
request b's query at position pos attends keys j <= pos with pos - j < W
when a window W is set."""
import numpy as np
import pytest

import bench
from paged_kv_gqa_12_gb300 import workloads as wl


def _attended(pos, window):
    return [j for j in range(pos + 1) if window <= 0 or pos - j < window]


@pytest.mark.parametrize("window", [0, 1, 7, 40])
def test_extend_flops_counts_attended_pairs(window):
    ctx = [0, 5, 37, 100]
    ql = [9, 1, 20, 3]
    p = wl.build_problem("extend", num_q_heads=6, num_kv_heads=2, head_dim=16, page_size=4,
                         seq_lens=np.array(ctx) + np.array(ql), query_lens=ql, window=window, seed=1)
    pairs = sum(len(_attended(c + i, window)) for c, q in zip(ctx, ql) for i in range(q))
    assert bench.extend_flops(p) == 4 * 16 * 6 * pairs


@pytest.mark.parametrize("kv,window", [("bf16", 0), ("bf16", 9), ("fp8_e4m3", 13), ("fp8_e4m3", 0)])
def test_decode_bytes_counts_attended_keys_and_pages(kv, window):
    lens = [1, 4, 5, 30, 64, 0]
    extra = dict(k_scale=0.1, v_scale=0.1) if kv == "fp8_e4m3" else {}
    p = wl.build_problem("decode", num_q_heads=8, num_kv_heads=2, head_dim=16, page_size=4,
                         seq_lens=lens, window=window, kv_dtype=kv, seed=2, **extra)
    e = 1 if kv == "fp8_e4m3" else 2
    keys = pages = 0
    for L in lens:
        J = _attended(L - 1, window) if L > 0 else []
        keys += len(J)
        pages += len({j // 4 for j in J})
    want = keys * 2 * 16 * e * 2 + len(lens) * 8 * 16 * 2 * 2 + len(lens) * 8 * 4 + pages * 4
    assert bench.decode_bytes(p) == want


def test_decode_plan_arguments_follow_the_workload():
    from paged_kv_gqa_12_gb300 import binding as pb
    tiny = wl.workload_problem("decode_tiny")
    assert bench.decode_plan_kw(pb, tiny, "decode_tiny")["num_splits"] == 4
    assert bench.decode_plan_kw(pb, tiny, "decode_tiny", splits=2)["num_splits"] == 2
    e4 = wl.workload_problem("decode_e4m3_window", batch=2)
    kw = bench.decode_plan_kw(pb, e4, "decode_e4m3_window")
    assert kw["kv_dtype"] == pb.KV_FP8_E4M3 and kw["window"] == 1024 and kw["has_sinks"] and kw["num_splits"] == 0


def test_clock_summary_marks_its_window():
    # samples inside the timed window are summarised as such; with none
    # inside, the record says it falls back to the whole run
    import bench
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.max_mhz, s.source = 2070.0, "test"
    s.samples = [(1.0, 2070.0, 500.0, []), (2.0, 1900.0, 900.0, ["sw_power_cap"]), (3.0, 2070.0, 600.0, [])]
    inside = s.summary(1.5, 2.5)
    assert inside["window"] == "timed region" and inside["samples"] == 1
    assert inside["sm_mhz"] == 1900.0 and inside["reasons"] == ["sw_power_cap"]
    outside = s.summary(10.0, 10.01)
    assert outside["window"].startswith("whole run") and outside["samples"] == 3
