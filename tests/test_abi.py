"""The C-ABI library: it builds, loads, exports every symbol include/*.h
declares, and its host-side logic (planning, argument checks) behaves, all
without a GPU."""
import ctypes
import glob
import os
import re

import pytest

from paged_kv_gqa_12_gb300 import binding as pb
from paged_kv_gqa_12_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return pb.load()


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names |= set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w]*\s*\**\s*(pa_\w+)\s*\(", src, flags=re.M))
    return names


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert {"pa_plan", "pa_decode", "pa_extend", "pa_check", "pa_scratch_init"} <= names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
    assert set(pb.EXPORTED_SYMBOLS) <= names


def test_version_and_strings(lib):
    assert lib.pa_version() >= 100
    for s in range(6):
        assert pb.status_string(s)


def _plan(**kw):
    base = dict(mode=pb.MODE_DECODE, num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                max_batch=64, max_pages_per_seq=512, num_sms=152)
    base.update(kw)
    return pb.plan(**base)


def test_plan_decode_defaults(lib):
    p = _plan()
    assert p.tile_tokens in (16, 32, 64)
    assert p.max_splits >= 1 and p.split_tiles >= 1
    assert p.grid[0] == p.max_splits and p.grid[1] == 8 and p.grid[2] == 64
    assert p.scratch_bytes >= pb.SCRATCH_HEADER_BYTES + 64 * 32 * p.max_splits * (128 + 1) * 4
    assert p.smem_bytes <= 232448


def test_scratch_layout_matches_binding_constants(lib):
    # header (error word + arrival counters), then o_part [B, Hq, S, D] and
    # lse_part [B, Hq, S] fp32, each rounded up to 256 bytes
    p = _plan(num_splits=3)
    o_part = 64 * 32 * 3 * 128 * 4
    lse_part = -(-(64 * 32 * 3 * 4) // 256) * 256
    assert p.scratch_bytes == pb.SCRATCH_HEADER_BYTES + o_part + lse_part
    assert pb.MERGE_COUNTERS == (pb.SCRATCH_HEADER_BYTES - 256) // 4


def test_plan_uses_host_lengths(lib):
    short = _plan(host_seq_lens=[600] * 64)
    long = _plan(host_seq_lens=[8000] * 64)
    assert long.split_tiles >= short.split_tiles


def test_plan_fixed_splits(lib):
    p = _plan(num_splits=4, max_pages_per_seq=19)
    assert p.max_splits == 4 and p.split_tiles == 0


@pytest.mark.parametrize("bad,status", [
    (dict(num_q_heads=30), pb.PA_ERR_INVALID_ARG),         # Hq % Hkv != 0
    (dict(head_dim=96), pb.PA_ERR_UNSUPPORTED),
    (dict(page_size=8), pb.PA_ERR_UNSUPPORTED),
    (dict(num_q_heads=129 * 8, num_kv_heads=8), pb.PA_ERR_UNSUPPORTED),  # group 129
    (dict(window=-1), pb.PA_ERR_INVALID_ARG),
    (dict(soft_cap=-1.0), pb.PA_ERR_INVALID_ARG),
    (dict(soft_cap=float("inf")), pb.PA_ERR_INVALID_ARG),
    (dict(kv_dtype=7), pb.PA_ERR_INVALID_ARG),
    (dict(mode=5), pb.PA_ERR_INVALID_ARG),
    (dict(host_seq_lens=[10, -1]), pb.PA_ERR_INVALID_ARG),
    (dict(host_seq_lens=[512 * 16 + 1]), pb.PA_ERR_INVALID_ARG),
])
def test_plan_rejects(lib, bad, status):
    with pytest.raises(pb.PaError) as ei:
        _plan(**bad)
    assert ei.value.status == status


def _decode_args(plan, **over):
    a = dict(plan=plan, q=0x10000, qs=(32 * 128, 128), k=0x20000, v=0x40000, kvs=(16 * 8 * 128, 8 * 128, 128),
             pages=100, bt=0x50000, bts=512, sl=0x60000, batch=4, scale=0.088, sinks=None, ks=1.0, vs=1.0,
             out=0x70000, os=(32 * 128, 128), lse=None, scratch=0x100000, sbytes=plan.scratch_bytes, stream=None)
    a.update(over)
    L = pb.load()
    vp = ctypes.c_void_p
    return L.pa_decode(ctypes.byref(a["plan"]), vp(a["q"]), a["qs"][0], a["qs"][1], vp(a["k"]), vp(a["v"]),
                       a["kvs"][0], a["kvs"][1], a["kvs"][2], a["pages"], vp(a["bt"]), a["bts"], vp(a["sl"]),
                       a["batch"], a["scale"], vp(a["sinks"]) if a["sinks"] else None, a["ks"], a["vs"], None, None,
                       vp(a["out"]), a["os"][0], a["os"][1], vp(a["lse"]) if a["lse"] else None,
                       vp(a["scratch"]) if a["scratch"] else None, a["sbytes"], None)


@pytest.mark.parametrize("over,status", [
    (dict(batch=65), pb.PA_ERR_INVALID_ARG),
    (dict(batch=-1), pb.PA_ERR_INVALID_ARG),
    (dict(sbytes=255), pb.PA_ERR_SCRATCH_TOO_SMALL),
    (dict(scratch=0), pb.PA_ERR_INVALID_ARG),
    (dict(scratch=0x100010), pb.PA_ERR_UNSUPPORTED),        # scratch not 256-byte aligned
    (dict(sinks=0x80000), pb.PA_ERR_INVALID_ARG),           # plan has no sinks
    (dict(scale=float("nan")), pb.PA_ERR_INVALID_ARG),
    (dict(q=0), pb.PA_ERR_INVALID_ARG),
    (dict(q=0x10002), pb.PA_ERR_UNSUPPORTED),               # q not 4-byte aligned
    (dict(k=0x20008), pb.PA_ERR_UNSUPPORTED),               # cache not 16-byte aligned
    (dict(kvs=(16 * 8 * 128, 8 * 128 + 4, 128)), pb.PA_ERR_UNSUPPORTED),  # token stride not 16B multiple
    (dict(pages=0), pb.PA_ERR_INVALID_ARG),
    (dict(bt=0), pb.PA_ERR_INVALID_ARG),
    (dict(out=0), pb.PA_ERR_INVALID_ARG),
])
def test_decode_rejects_before_launch(lib, over, status):
    plan = _plan()
    assert _decode_args(plan, **over) == status


def test_decode_rejects_hand_edited_plans(lib):
    # split_merge set on a plan whose pairs exceed the header's counters, or a
    # scratch size below the header: refused before anything is enqueued
    plan = _plan(max_batch=pb.MERGE_COUNTERS // 8 + 1, num_splits=2)
    assert plan.split_merge == 0
    plan.split_merge = 1
    assert _decode_args(plan) == pb.PA_ERR_INVALID_ARG
    small = _plan(num_splits=1)
    small.scratch_bytes = 4096
    assert _decode_args(small, sbytes=4096) == pb.PA_ERR_SCRATCH_TOO_SMALL
    # more splits (or a larger shape) than scratch_bytes was computed for: the
    # partials would run past the buffer, so the plan is refused
    more = _plan(num_splits=3)
    more.max_splits = 5
    more.grid[0] = 5
    assert _decode_args(more) == pb.PA_ERR_INVALID_ARG
    wider = _plan(num_splits=3)
    wider.shape.max_batch = 128
    assert _decode_args(wider) == pb.PA_ERR_INVALID_ARG
    none = _plan(num_splits=3)
    none.max_splits = 0
    assert _decode_args(none) == pb.PA_ERR_INVALID_ARG
    tile = _plan()
    tile.tile_tokens *= 2
    assert _decode_args(tile) == pb.PA_ERR_INVALID_ARG


def _extend_args(plan, sbytes=None, batch=4, total_q=64):
    L = pb.load()
    vp = ctypes.c_void_p
    return L.pa_extend(ctypes.byref(plan), vp(0x10000), 32 * 128, 128, vp(0x20000), vp(0x40000), 16 * 8 * 128,
                       8 * 128, 128, 100, vp(0x50000), 512, vp(0x60000), vp(0x68000), batch, total_q, 0.088, None,
                       1.0, 1.0, None, None, vp(0x70000), 32 * 128, 128, None, vp(0x100000),
                       plan.scratch_bytes if sbytes is None else sbytes, None)


def test_extend_rejects_hand_edited_plans(lib):
    # the work list (and an e4m3 copy) are laid out from the shape's
    # capacities: a plan whose grid or scratch size no longer matches them
    # is refused before anything is enqueued
    try:
        base = _plan(mode=pb.MODE_EXTEND, max_total_q=1024, max_batch=8)
    except pb.PaError:
        pytest.skip("extend planning unavailable")
    grid = _plan(mode=pb.MODE_EXTEND, max_total_q=1024, max_batch=8)
    grid.grid[0] += 8
    assert _extend_args(grid) == pb.PA_ERR_INVALID_ARG
    fp8 = _plan(mode=pb.MODE_EXTEND, max_total_q=1024, max_batch=8, kv_dtype=pb.KV_FP8_E4M3)
    assert fp8.kv_copy == 1
    full = fp8.scratch_bytes
    fp8.scratch_bytes = base.scratch_bytes   # the copy's room edited away
    assert _extend_args(fp8, sbytes=base.scratch_bytes) == pb.PA_ERR_SCRATCH_TOO_SMALL
    assert _extend_args(fp8, sbytes=full - 256) == pb.PA_ERR_SCRATCH_TOO_SMALL
    # the unedited plans pass these checks (empty calls: nothing to launch)
    assert _extend_args(base, batch=0, total_q=0) == pb.PA_OK
    fp8.scratch_bytes = full
    assert _extend_args(fp8, batch=0, total_q=0) == pb.PA_OK


def test_decode_empty_batch_is_noop(lib):
    plan = _plan()
    assert _decode_args(plan, batch=0) == pb.PA_OK


def test_decode_rejects_extend_plan(lib):
    try:
        plan = _plan(mode=pb.MODE_EXTEND, max_total_q=1024)
    except pb.PaError:
        pytest.skip("extend planning unavailable")
    assert _decode_args(plan) == pb.PA_ERR_INVALID_ARG


def test_binding_fails_loudly_without_library(tmp_path):
    import importlib
    b2 = importlib.reload(pb)
    try:
        b2._lib = None
        with pytest.raises(RuntimeError):
            b2.load(str(tmp_path / "missing.so"))
    finally:
        importlib.reload(pb)


@pytest.mark.parametrize("q_len,status", [(0, pb.PA_ERR_INVALID_ARG), (5, pb.PA_ERR_UNSUPPORTED)])
def test_plan_verify_rejects(lib, q_len, status):
    # 32 q heads over 8 kv heads: group 4, so at most 4 tokens per request
    with pytest.raises(pb.PaError) as ei:
        _plan(mode=pb.MODE_VERIFY, q_len=q_len, max_total_q=256)
    assert ei.value.status == status


def test_plan_verify_scratch_scales_with_q_len(lib):
    one = _plan(mode=pb.MODE_VERIFY, q_len=1, max_total_q=64, num_splits=4)
    four = _plan(mode=pb.MODE_VERIFY, q_len=4, max_total_q=256, num_splits=4)
    h = pb.SCRATCH_HEADER_BYTES
    assert four.scratch_bytes - h > 3 * (one.scratch_bytes - h)
    assert four.split_merge == 1 and four.launches == 1


def test_plan_extend_e4m3_copy_choice(lib):
    # an e4m3 extend plan dequantises into a bf16 copy while that copy
    # (max_batch x max_pages_per_seq pages, K and V) fits in 2 GiB
    kw = dict(mode=pb.MODE_EXTEND, kv_dtype=pb.KV_FP8_E4M3, max_batch=8, max_total_q=4096)
    small = _plan(max_pages_per_seq=384, **kw)
    copy_bytes = 8 * 384 * 16 * 8 * 128 * 2 * 2
    assert small.kv_copy == 1 and small.launches == 3
    bf16 = _plan(mode=pb.MODE_EXTEND, max_batch=8, max_total_q=4096, max_pages_per_seq=384)
    assert bf16.kv_copy == 0 and bf16.launches == 2
    assert small.scratch_bytes >= bf16.scratch_bytes + copy_bytes + 8 * 384 * 4
    big = _plan(max_pages_per_seq=1 << 16, **kw)
    assert big.kv_copy == 0 and big.launches == 2 and big.scratch_bytes < (1 << 20)


def test_plan_single_split_makes_one_launch(lib):
    # one split per request: the split kernel writes the outputs, no merge launch
    one = _plan(num_splits=1)
    assert one.max_splits == 1 and one.launches == 1 and one.split_merge == 0


def test_plan_split_merge_follows_counter_capacity(lib):
    # several splits: the last split of each (request, kv head) merges while the
    # scratch header has a counter per pair; beyond that a merge kernel follows
    two = _plan(num_splits=2)
    assert two.split_merge == 1 and two.launches == 1
    fits = _plan(num_splits=2, max_batch=pb.MERGE_COUNTERS // 8)
    assert fits.split_merge == 1 and fits.launches == 1
    over = _plan(num_splits=2, max_batch=pb.MERGE_COUNTERS // 8 + 1)
    assert over.split_merge == 0 and over.launches == 2
    # head groups count: group 32 over 2 kv heads is 4 pairs per request
    g = _plan(num_splits=2, num_q_heads=64, num_kv_heads=2, max_batch=pb.MERGE_COUNTERS // 4 + 1)
    assert g.split_merge == 0 and g.launches == 2


def test_plan_decode_large_group_uses_head_groups(lib):
    p = _plan(num_q_heads=64, num_kv_heads=2)          # group 32: two CTAs of 16 heads per kv head
    assert p.grid[1] == 2 * 2
    q = _plan(num_q_heads=40, num_kv_heads=2)          # group 20: 16 + 4
    assert q.grid[1] == 2 * 2
    e = _plan(mode=pb.MODE_EXTEND, num_q_heads=128, num_kv_heads=1, max_total_q=512)
    assert e.launches == 2


def test_debug_wait_expiry_rejects_before_launch(lib):
    vp = ctypes.c_void_p
    L = pb.load()
    assert L.pa_debug_wait_expiry(None, 0, 2_000_000, None) == pb.PA_ERR_INVALID_ARG
    assert L.pa_debug_wait_expiry(vp(0x100000), 5, 2_000_000, None) == pb.PA_ERR_INVALID_ARG
    assert L.pa_debug_wait_expiry(vp(0x100000), 0, 999, None) == pb.PA_ERR_INVALID_ARG
    assert L.pa_debug_wait_expiry(vp(0x100000), 0, 10**8 + 1, None) == pb.PA_ERR_INVALID_ARG
    assert L.pa_debug_wait_expiry(vp(0x100010), 0, 2_000_000, None) == pb.PA_ERR_UNSUPPORTED


def test_device_code_bits_match_header(lib):
    src = open(os.path.join(ROOT, "include", "pa.h")).read()
    for name, val in (("WAIT_TIMEOUT", pb.DEVICE_WAIT_TIMEOUT), ("WORK_OVERFLOW", pb.DEVICE_WORK_OVERFLOW),
                      ("CAPACITY", pb.DEVICE_CAPACITY), ("PAGE_ID", pb.DEVICE_PAGE_ID)):
        m = re.search(r"PA_DEVICE_%s\s*=\s*(\d+)" % name, src)
        assert m and int(m.group(1)) == val, name
