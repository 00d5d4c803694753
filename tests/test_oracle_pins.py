"""Pins of the CPU oracle against things other than itself.

Each test names what it pins; together they are chosen so that a plausible
slip in the oracle (a dropped scale, a transposed head map, a wrong page or
slot index, a window off by one, soft-cap before scaling, a sink given a value
row, a mis-decoded fp8 code) fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_gqa_12_gb300 import workloads as wl
from tests import refs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _problem(mode="decode", seed=0, B=3, Hq=4, Hkv=2, D=8, ps=4, lens=None, qlens=None, **kw):
    rng = np.random.default_rng(seed + 17)
    if lens is None:
        lens = rng.integers(1, 41, size=B)
    if mode == "extend" and qlens is None:
        qlens = np.minimum(rng.integers(1, 13, size=B), lens)
    return wl.build_problem(mode, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=ps,
                            seq_lens=lens, query_lens=qlens, seed=seed, keep_logical=True, **kw)


def _rows_of(p, b):
    if p.mode == "decode":
        return [b]
    return list(range(int(p.query_start_loc[b]), int(p.query_start_loc[b + 1])))


# ---- element decoding: library routines ---------------------------------------

def test_bf16_decode_all_codes(oracle_lib):
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = refs.bf16_bits_to_f64(codes).numpy()
    got = np.array([oracle.bf16_to_double(c) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])


def test_e4m3_decode_all_codes(oracle_lib):
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle.e4m3_to_double(c) for c in codes])
    nan = np.isnan(ref)
    assert nan.sum() == 2                      # S.1111.111 only
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])


def test_e4m3_golden_values(oracle_lib):
    # tests/golden/e4m3_format.txt: landmark codes of the OCP FP8 E4M3 format.
    with open(os.path.join(GOLDEN, "e4m3_format.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    assert len(rows) >= 8
    for code, val in rows:
        v = oracle.e4m3_to_double(int(code, 16))
        if val == "nan":
            assert math.isnan(v)
        else:
            assert v == float.fromhex(val), (code, val, v)


@pytest.mark.parametrize("scale", [0.05, 1.0, 0.3, 3.75, 1e-3])
def test_fp8_dequant_all_codes(oracle_lib, scale):
    codes = np.arange(256, dtype=np.uint8)
    ref = refs.e4m3_dequant_f64(codes, scale).numpy()
    got = np.array([oracle.fp8_dequant(c, scale) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])


# ---- brute force: torch SDPA on the logical (unpaged) K/V ---------------------

CASES = [
    # mode,   G, Hkv, D,  ps, layout,        kv
    ("decode", 1, 2, 8, 1, "separate", "bf16"),
    ("decode", 4, 2, 8, 4, "interleaved", "bf16"),
    ("decode", 2, 1, 64, 16, "separate", "bf16"),
    ("decode", 4, 2, 16, 4, "separate", "fp8_e4m3"),
    ("extend", 1, 1, 8, 1, "separate", "bf16"),
    ("extend", 4, 2, 8, 4, "interleaved", "bf16"),
    ("extend", 2, 2, 64, 16, "separate", "bf16"),
    ("extend", 8, 1, 16, 8, "separate", "fp8_e4m3"),
]


@pytest.mark.parametrize("mode,G,Hkv,D,ps,layout,kv", CASES)
def test_oracle_matches_sdpa(oracle_lib, mode, G, Hkv, D, ps, layout, kv):
    extra = dict(kv_dtype=kv, layout=layout)
    if kv == "fp8_e4m3":
        extra.update(k_scale=0.05, v_scale=0.07)
    p = _problem(mode, seed=G * 100 + D + ps, Hq=G * Hkv, Hkv=Hkv, D=D, ps=ps, **extra)
    out, lse = oracle.attention(p)
    q = refs.bf16_bits_to_f64(p.q)
    for b in range(p.batch):
        rows = _rows_of(p, b)
        k, v = refs.logical_kv_f64(p, b)
        keep = refs.lower_right_causal(len(rows), int(p.seq_lens[b]))
        O, LSE = refs.sdpa_with_lse(q[rows], k, v, keep, p.scale)
        np.testing.assert_allclose(out[rows], O.numpy(), rtol=0, atol=1e-11)
        np.testing.assert_allclose(lse[rows], LSE.numpy(), rtol=0, atol=1e-11)


@pytest.mark.parametrize("mode", ["decode", "extend"])
def test_oracle_per_request_scales_match_sdpa(oracle_lib, mode):
    # per-request e4m3 descales (the b12x backend's [num_reqs] descale
    # tensors): each request's logical K/V dequantised with its own scales
    ks, vs = [0.05, 0.11, 0.02], [0.07, 0.013, 0.3]
    p = _problem(mode, seed=811, Hq=8, Hkv=2, D=16, ps=4, kv_dtype="fp8_e4m3", k_scales=ks, v_scales=vs)
    out, lse = oracle.attention(p)
    q = refs.bf16_bits_to_f64(p.q)
    for b in range(p.batch):
        rows = _rows_of(p, b)
        k, v = refs.logical_kv_f64(p, b)
        keep = refs.lower_right_causal(len(rows), int(p.seq_lens[b]))
        O, LSE = refs.sdpa_with_lse(q[rows], k, v, keep, p.scale)
        np.testing.assert_allclose(out[rows], O.numpy(), rtol=0, atol=1e-11)
        np.testing.assert_allclose(lse[rows], LSE.numpy(), rtol=0, atol=1e-11)


def test_per_request_scales_equal_to_scalar(oracle_lib):
    # the same scale for every request is the per-tensor case, bit for bit
    a = _problem("extend", seed=812, kv_dtype="fp8_e4m3", k_scale=0.05, v_scale=0.07)
    b = _problem("extend", seed=812, kv_dtype="fp8_e4m3", k_scales=[0.05] * 3, v_scales=[0.07] * 3)
    assert np.array_equal(a.k_cache, b.k_cache) and np.array_equal(a.v_cache, b.v_cache)
    oa, la = oracle.attention(a)
    ob, lb = oracle.attention(b)
    assert np.array_equal(oa, ob) and np.array_equal(la, lb)


def test_per_request_scales_follow_the_request(oracle_lib):
    # each request of a mixed batch equals that request alone with its own
    # scalar scales, over the same pages (a scale taken from the wrong request
    # or row fails here)
    import dataclasses
    ks, vs = [0.05, 0.11, 0.02], [0.07, 0.013, 0.3]
    p = _problem("extend", seed=813, kv_dtype="fp8_e4m3", k_scales=ks, v_scales=vs)
    out, lse = oracle.attention(p)
    qsl = p.query_start_loc
    for b in range(p.batch):
        r0, r1 = int(qsl[b]), int(qsl[b + 1])
        one = dataclasses.replace(p, q=p.q[r0:r1], block_table=p.block_table[b:b + 1],
                                  seq_lens=p.seq_lens[b:b + 1], query_start_loc=np.array([0, r1 - r0], np.int32),
                                  k_scales=None, v_scales=None, k_scale=ks[b], v_scale=vs[b])
        o1, l1 = oracle.attention(one)
        assert np.array_equal(o1, out[r0:r1]) and np.array_equal(l1, lse[r0:r1]), b


# ---- closed forms -----------------------------------------------------------

def test_single_key_is_value_row(oracle_lib):
    p = _problem("decode", seed=5, B=4, lens=[1, 1, 1, 1], Hq=8, Hkv=2, D=16, ps=4)
    out, lse = oracle.attention(p)
    q = refs.bf16_bits_to_f64(p.q)
    for b in range(4):
        k, v = refs.logical_kv_f64(p, b)
        for h in range(8):
            kvh = h // 4
            assert np.array_equal(out[b, h], v[0, kvh].numpy())  # O = V_0 exactly
            s = p.scale * float((q[b, h] * k[0, kvh]).sum())
            assert abs(lse[b, h] - s) < 1e-12


@pytest.mark.parametrize("sinks", [False, True])
@pytest.mark.parametrize("window", [0, 1, 5, 17])
def test_zero_query_is_mean_of_window(oracle_lib, window, sinks):
    # q = 0 makes every score 0: O = sum of the attended V rows / (|J| + e^sink),
    # LSE = ln(|J| + e^sink), with |J| = min(window, pos+1) most recent keys.
    for mode in ("decode", "extend"):
        p = _problem(mode, seed=11 + window, B=3, Hq=4, Hkv=2, D=8, ps=4,
                     lens=[9, 30, 40], qlens=[3, 7, 1] if mode == "extend" else None,
                     window=window, sinks=sinks, q_values=np.zeros((11 if mode == "extend" else 3, 4, 8), np.float32))
        out, lse = oracle.attention(p)
        for b in range(p.batch):
            k, v = refs.logical_kv_f64(p, b)
            L = int(p.seq_lens[b])
            rows = _rows_of(p, b)
            for i, r in enumerate(rows):
                pos = L - len(rows) + i
                lo = 0 if window <= 0 else max(0, pos - window + 1)
                n = pos + 1 - lo
                for h in range(4):
                    extra = math.exp(float(p.sinks[h])) if sinks else 0.0
                    Z = n + extra
                    ref_o = v[lo:pos + 1, h // 2].sum(0).numpy() / Z
                    np.testing.assert_allclose(out[r, h], ref_o, rtol=0, atol=1e-12)
                    assert abs(lse[r, h] - math.log(Z)) < 1e-12


def test_window_one_is_identity(oracle_lib):
    # window = 1: every query attends to itself only -> O = V_pos exactly.
    p = _problem("extend", seed=3, B=2, Hq=4, Hkv=2, D=8, ps=4, lens=[13, 22], qlens=[13, 5], window=1)
    out, _ = oracle.attention(p)
    for b in range(2):
        k, v = refs.logical_kv_f64(p, b)
        L = int(p.seq_lens[b])
        rows = _rows_of(p, b)
        for i, r in enumerate(rows):
            pos = L - len(rows) + i
            for h in range(4):
                assert np.array_equal(out[r, h], v[pos, h // 2].numpy())


def test_softcap_applied_after_scale(oracle_lib):
    # One key, score scale*q.k = ln 3, cap = 2: cap*tanh(ln3/2) = 1 exactly.
    # Capping before scaling would give scale*2*tanh(q.k/2) = 0.8 here.
    a, bval = 2.0, 1.5
    qv = np.zeros((1, 1, 8), np.float32)
    qv[0, 0, 0] = a
    p = _problem("decode", seed=1, B=1, Hq=1, Hkv=1, D=8, ps=4, lens=[1], q_values=qv)
    p.logical_k[0][0, 0, :] = 0
    p.logical_k[0][0, 0, 0] = wl._to_bf16_bits(np.array([bval], np.float32))[0]
    p.k_cache[p.block_table[0, 0], 0, 0, :] = p.logical_k[0][0, 0, :]
    p.scale = math.log(3.0) / (a * bval)
    p.soft_cap = 2.0
    _, lse = oracle.attention(p)
    assert abs(lse[0, 0] - 1.0) < 1e-12
    p.soft_cap = 0.0
    _, lse0 = oracle.attention(p)
    assert abs(lse0[0, 0] - math.log(3.0)) < 1e-12


def test_softcap_bounds_and_huge_cap(oracle_lib):
    p = _problem("decode", seed=9, B=3, Hq=4, Hkv=2, D=64, ps=4)
    out0, lse0 = oracle.attention(p)
    p.soft_cap = 1e30
    out1, lse1 = oracle.attention(p)
    np.testing.assert_allclose(out1, out0, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse1, lse0, rtol=0, atol=1e-13)
    # every capped logit lies in (-cap, cap): LSE <= ln|J| + cap
    p.soft_cap = 0.25
    _, lse2 = oracle.attention(p)
    for b in range(3):
        assert np.all(lse2[b] <= math.log(int(p.seq_lens[b])) + 0.25)
        assert np.all(lse2[b] >= math.log(int(p.seq_lens[b])) - 0.25)


def test_sink_minus_infinity_is_no_sink(oracle_lib):
    p = _problem("decode", seed=21, B=3, Hq=4, Hkv=2, D=8, ps=4)
    out0, lse0 = oracle.attention(p)
    p.sinks = np.full(4, -1e30, np.float32)
    out1, lse1 = oracle.attention(p)
    assert np.array_equal(out0, out1) and np.array_equal(lse0, lse1)


def test_sink_identity_relation(oracle_lib):
    # With a sink, LSE includes it: sum_j e^(s_j - LSE) = 1 - e^(sink - LSE), and
    # O is the no-sink output scaled by that mass.
    p = _problem("decode", seed=22, B=3, Hq=4, Hkv=2, D=8, ps=4)
    out0, lse0 = oracle.attention(p)
    p.sinks = np.array([0.5, -1.0, 2.0, 0.0], np.float32)
    out1, lse1 = oracle.attention(p)
    mass = 1.0 - np.exp(p.sinks[None, :].astype(np.float64) - lse1)
    np.testing.assert_allclose(np.exp(lse0 - lse1), mass, rtol=1e-12)
    np.testing.assert_allclose(out1, out0 * mass[..., None], rtol=0, atol=1e-13)


# ---- invariances --------------------------------------------------------------

def _permute_pages(p, seed):
    rng = np.random.default_rng(seed)
    P = p.num_pages
    perm = rng.permutation(P)               # new location of old page i is perm[i]
    k2 = np.empty_like(p.k_cache)
    v2 = np.empty_like(p.v_cache)
    k2[perm] = p.k_cache
    v2[perm] = p.v_cache
    bt = p.block_table.copy()
    used = bt != wl.BT_SENTINEL
    bt[used] = perm[bt[used]]
    import dataclasses
    return dataclasses.replace(p, k_cache=k2, v_cache=v2, block_table=bt, kv_storage=None)


@pytest.mark.parametrize("mode", ["decode", "extend"])
def test_page_permutation_invariance(oracle_lib, mode):
    p = _problem(mode, seed=31, B=4, Hq=8, Hkv=2, D=16, ps=4, window=7, sinks=True, soft_cap=3.0)
    out0, lse0 = oracle.attention(p)
    out1, lse1 = oracle.attention(_permute_pages(p, 5))
    assert np.array_equal(out0, out1) and np.array_equal(lse0, lse1)


def test_layout_invariance(oracle_lib):
    a = _problem("extend", seed=41, B=3, Hq=4, Hkv=2, D=8, ps=4, layout="separate")
    b = _problem("extend", seed=41, B=3, Hq=4, Hkv=2, D=8, ps=4, layout="interleaved")
    oa, la = oracle.attention(a)
    ob, lb = oracle.attention(b)
    assert np.array_equal(oa, ob) and np.array_equal(la, lb)


def test_window_at_least_length_is_no_window(oracle_lib):
    p = _problem("extend", seed=51, B=3, Hq=4, Hkv=2, D=8, ps=4, lens=[10, 25, 40], qlens=[4, 25, 2])
    o0, l0 = oracle.attention(p)
    p.window = 40
    o1, l1 = oracle.attention(p)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)


def test_window_equals_suffix_sequence(oracle_lib):
    # Decode with window W over a length-L sequence = decode without window
    # over a fresh length-W sequence made of the last W tokens.
    p = _problem("decode", seed=61, B=2, Hq=4, Hkv=2, D=8, ps=4, lens=[37, 23], window=9)
    o, l = oracle.attention(p)
    W = 9
    sufk = [lk[-W:] for lk in p.logical_k]
    sufv = [lv[-W:] for lv in p.logical_v]
    s = wl.build_problem("decode", num_q_heads=4, num_kv_heads=2, head_dim=8, page_size=4,
                         seq_lens=[W, W], seed=62, keep_logical=True)
    for b in range(2):
        for t in range(W):
            s.k_cache[s.block_table[b, t // 4], t % 4] = sufk[b][t]
            s.v_cache[s.block_table[b, t // 4], t % 4] = sufv[b][t]
    s.q = p.q.copy()
    s.scale = p.scale
    o2, l2 = oracle.attention(s)
    assert np.array_equal(o, o2) and np.array_equal(l, l2)


@pytest.mark.parametrize("cap", [0.0, 5.0])
def test_split_and_lse_merge_reproduce_the_whole(oracle_lib, cap):
    # Split-KV is an exact re-association: attention over keys [0, a) and over
    # [a, L), merged by their log-sum-exps, is attention over [0, L).  The two
    # parts come from the oracle itself, through its own definition: the first
    # a keys are the request with seq_len a (same query, same pages), the last
    # L - a keys are the request with window L - a.  The merge is written
    # here in float64: M = max(lse1, lse2), w_i = exp(lse_i - M),
    # O = (w1 O1 + w2 O2) / (w1 + w2), LSE = M + ln(w1 + w2).
    import dataclasses
    W = 9
    p = _problem("decode", seed=66, B=3, Hq=8, Hkv=2, D=16, ps=4, lens=[37, 23, 41], soft_cap=cap)
    o, l = oracle.attention(p)
    head = dataclasses.replace(p, seq_lens=p.seq_lens - W)
    tail = dataclasses.replace(p, window=W)
    o1, l1 = oracle.attention(head)
    o2, l2 = oracle.attention(tail)
    M = np.maximum(l1, l2)
    w1, w2 = np.exp(l1 - M), np.exp(l2 - M)
    om = (w1[..., None] * o1 + w2[..., None] * o2) / (w1 + w2)[..., None]
    lm = M + np.log(w1 + w2)
    assert np.abs(om - o).max() <= 1e-12
    assert np.abs(lm - l).max() <= 1e-12


def test_extend_single_query_equals_decode(oracle_lib):
    e = _problem("extend", seed=71, B=3, Hq=8, Hkv=2, D=16, ps=4, lens=[5, 19, 33], qlens=[1, 1, 1],
                 window=6, sinks=True, soft_cap=4.0)
    oe, le = oracle.attention(e)
    import dataclasses
    d = dataclasses.replace(e, mode="decode", query_start_loc=None)
    od, ld = oracle.attention(d)
    assert np.array_equal(oe, od) and np.array_equal(le, ld)


def test_chunked_extend_matches_whole(oracle_lib):
    # Extending by q1+q2 tokens at once gives, for the last q2 rows, exactly the
    # rows of a second extend of q2 tokens whose context already holds q1.
    whole = _problem("extend", seed=81, B=2, Hq=4, Hkv=2, D=8, ps=4, lens=[30, 21], qlens=[12, 9])
    ow, lw = oracle.attention(whole)
    import dataclasses
    q2 = np.array([5, 4])
    starts = whole.query_start_loc
    sel = np.concatenate([np.arange(starts[b + 1] - q2[b], starts[b + 1]) for b in range(2)])
    second = dataclasses.replace(whole, q=whole.q[sel].copy(),
                                 query_start_loc=np.array([0, 5, 9], np.int32))
    o2, l2 = oracle.attention(second)
    assert np.array_equal(ow[sel], o2) and np.array_equal(lw[sel], l2)


def test_row_subset_matches_full(oracle_lib):
    p = _problem("extend", seed=91, B=3, Hq=4, Hkv=2, D=8, ps=4)
    o, l = oracle.attention(p)
    rows = np.array([0, p.num_rows - 1, p.num_rows // 2], np.int32)
    o2, l2 = oracle.attention(p, rows=rows)
    assert np.array_equal(o[rows], o2) and np.array_equal(l[rows], l2)


def test_poisoned_slots_never_read(oracle_lib):
    # The generator fills unreachable slots with NaN: finite results show the
    # oracle reads only the attended keys.
    p = _problem("extend", seed=101, B=3, Hq=4, Hkv=2, D=8, ps=8, window=5, sinks=True)
    o, l = oracle.attention(p)
    assert np.isfinite(o).all() and np.isfinite(l).all()
    assert np.isnan(refs.bf16_bits_to_f64(p.k_cache).numpy()).any()


def test_empty_sequence(oracle_lib):
    p = _problem("decode", seed=111, B=2, Hq=2, Hkv=1, D=8, ps=4, lens=[0, 3], sinks=True)
    o, l = oracle.attention(p)
    assert np.all(o[0] == 0.0)
    np.testing.assert_allclose(l[0], p.sinks.astype(np.float64), rtol=0, atol=0)
    p.sinks = None
    o, l = oracle.attention(p)
    assert np.all(o[0] == 0.0) and np.all(np.isneginf(l[0]))


def test_bad_block_table_rejected(oracle_lib):
    p = _problem("decode", seed=121, B=2, Hq=2, Hkv=1, D=8, ps=4, lens=[9, 3])
    p.block_table[0, 1] = p.num_pages + 3
    with pytest.raises(RuntimeError):
        oracle.attention(p)


# ---- the cache write side: e4m3 encoding and KV append ----------------------------

def test_e4m3_encode_roundtrips_every_code(oracle_lib):
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert oracle.e4m3_encode(oracle.e4m3_to_double(c)) == c, hex(c)


def test_e4m3_encode_matches_torch_including_ties(oracle_lib):
    # random values, every representable magnitude, and every midpoint between
    # neighbours (ties go to the even code), all inside the finite range
    rng = np.random.default_rng(5)
    vals = [float(x) for x in rng.uniform(-440, 440, 4000)] + [float(x) for x in rng.standard_normal(4000)]
    mags = sorted({oracle.e4m3_to_double(c) for c in range(0x7F)})
    vals += mags + [-m for m in mags] + [(a + b) / 2 for a, b in zip(mags, mags[1:])]
    x = torch.tensor(vals, dtype=torch.float32)
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(v) for v in x.numpy()], np.uint8)
    assert np.array_equal(ref, got)


def test_e4m3_encode_saturates_and_keeps_nan(oracle_lib):
    assert oracle.e4m3_encode(1e6) == 0x7E and oracle.e4m3_encode(-1e6) == 0xFE
    assert oracle.e4m3_encode(float("inf")) == 0x7E and oracle.e4m3_encode(464.0) == 0x7E
    assert oracle.e4m3_encode(float("nan")) & 0x7F == 0x7F


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
def test_append_kv_rebuilds_generated_cache(oracle_lib, kv):
    # Appending every token's K/V through the slot mapping reproduces the cache
    # the generator wrote (generator: torch's conversion; here: the oracle's).
    lens = [9, 30, 17]
    extra = dict(kv_dtype=kv, k_scale=0.05, v_scale=0.07) if kv == "fp8_e4m3" else {}
    base = _problem("decode", seed=131, B=3, Hq=4, Hkv=2, D=16, ps=4, lens=lens, **extra)
    # bf16 inputs whose quantisation the generator also performed
    rng = np.random.default_rng(9)
    ks, vs, slots = [], [], []
    for b, L in enumerate(lens):
        kx = wl._to_bf16_bits(rng.standard_normal((L, 2, 16), dtype=np.float32))
        vx = wl._to_bf16_bits(rng.standard_normal((L, 2, 16), dtype=np.float32))
        ks.append(kx)
        vs.append(vx)
        for t in range(L):
            slots.append(int(base.block_table[b, t // 4]) * 4 + t % 4)
    k_new, v_new = np.concatenate(ks), np.concatenate(vs)
    slots = np.array(slots + [-1, -7], np.int64)        # padding slots are skipped
    k_new = np.concatenate([k_new, k_new[:2]])
    v_new = np.concatenate([v_new, v_new[:2]])
    kc, vc = np.zeros_like(base.k_cache), np.zeros_like(base.v_cache)
    oracle.append_kv(k_new, v_new, kc, vc, slots, 0.05, 0.07)
    # reference: torch-based cache writes of the same values
    kr, vr = np.zeros_like(kc), np.zeros_like(vc)
    f32 = refs.bf16_bits_to_f64(k_new).float()
    g32 = refs.bf16_bits_to_f64(v_new).float()
    for t, s in enumerate(slots):
        if s < 0:
            continue
        if kv == "fp8_e4m3":
            kr[s // 4, s % 4] = (f32[t] / torch.tensor(0.05, dtype=torch.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            vr[s // 4, s % 4] = (g32[t] / torch.tensor(0.07, dtype=torch.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        else:
            kr[s // 4, s % 4] = k_new[t]
            vr[s // 4, s % 4] = v_new[t]
    assert np.array_equal(kc, kr) and np.array_equal(vc, vr)
    bad = slots.copy()
    bad[0] = kc.shape[0] * 4
    with pytest.raises(RuntimeError):
        oracle.append_kv(k_new, v_new, kc, vc, bad)
