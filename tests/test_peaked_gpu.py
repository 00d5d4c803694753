"""Parity on peaked attention: queries scaled up so that a few keys carry
almost all of each row's softmax weight, and soft-capped logits pressed
against the cap.  These rows do not average out the rounding of the softmax
weights over many keys, so they check that the kernels' weights stay within
the tolerances where the workloads' N(0,1) queries would not show it.

Operation: "vllm/attention/ops/triton_decode_attention.py" (decode, soft-cap
cap * tanh(s / cap) after scaling) and "vllm/attention/ops/prefix_prefill.py"
(extend).
"""
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


# (q multiplier, soft cap): peaked softmax; peaked and capped well above the
# typical logit; logits pressed against a low cap
PEAKS = [(6.0, 0.0), (8.0, 30.0), (8.0, 4.0)]


def _q(seed, rows, Hq, D, mult):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((rows, Hq, D)) * mult).astype(np.float32)


DECODE_SHAPES = [
    # Hq, Hkv, D, ps, kv
    (32, 8, 128, 16, "bf16"),
    (64, 8, 64, 64, "fp8_e4m3"),
    (16, 8, 256, 32, "bf16"),
]
LENS = [1, 2, 17, 200, 1500, 4100]


@pytest.mark.parametrize("Hq,Hkv,D,ps,kv", DECODE_SHAPES)
@pytest.mark.parametrize("mult,cap", PEAKS)
def test_decode_peaked(Hq, Hkv, D, ps, kv, mult, cap):
    extra = dict(k_scale=0.05, v_scale=0.05) if kv == "fp8_e4m3" else {}
    p = wl.build_problem("decode", num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=ps, seq_lens=LENS,
                         kv_dtype=kv, soft_cap=cap, seed=int(mult * 10 + cap + D), window=1000, sinks=True,
                         q_values=_q(D, len(LENS), Hq, D, mult), **extra)
    ref_o, ref_l = oracle.attention(p)
    for ns in (0, 1, 5):
        out, lse = gh.run(p, num_splits=ns)
        eo, el = gh.assert_parity(out, lse, ref_o, ref_l, what=f"peaked decode x{mult} cap {cap} splits {ns}")
        print(f"decode {Hq}/{Hkv}/{D} {kv} x{mult} cap {cap} splits {ns}: out {eo:.2e} lse {el:.2e}")


@pytest.mark.parametrize("mult,cap", PEAKS)
def test_verify_peaked(mult, cap):
    ctx = np.array([0, 3, 15, 700, 2047, 5000])
    ql = np.full_like(ctx, 4)
    p = wl.build_problem("extend", num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16, seq_lens=ctx + ql,
                         query_lens=ql, soft_cap=cap, seed=int(mult + cap) + 3,
                         q_values=_q(5, int(ql.sum()), 32, 128, mult))
    ref_o, ref_l = oracle.attention(p)
    out, lse = gh.run(p, verify=True)
    eo, el = gh.assert_parity(out, lse, ref_o, ref_l, what=f"peaked verify x{mult} cap {cap}")
    print(f"verify x{mult} cap {cap}: out {eo:.2e} lse {el:.2e}")


EXTEND_SHAPES = [(32, 8, 128, 16), (8, 2, 64, 16), (16, 8, 256, 32)]
CTX = [0, 5, 300, 1000, 129, 3000]
QL = [37, 1, 200, 64, 513, 300]


@pytest.mark.parametrize("Hq,Hkv,D,ps", EXTEND_SHAPES)
@pytest.mark.parametrize("mult,cap", PEAKS)
def test_extend_peaked(Hq, Hkv, D, ps, mult, cap):
    ctx, ql = np.array(CTX), np.array(QL)
    p = wl.build_problem("extend", num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=ps, seq_lens=ctx + ql,
                         query_lens=ql, soft_cap=cap, seed=int(mult * 3 + cap + D),
                         q_values=_q(D + 1, int(ql.sum()), Hq, D, mult))
    ref_o, ref_l = oracle.attention(p)
    out, lse = gh.run(p)
    eo, el = gh.assert_parity(out, lse, ref_o, ref_l, what=f"peaked extend x{mult} cap {cap}")
    print(f"extend {Hq}/{Hkv}/{D} x{mult} cap {cap}: out {eo:.2e} lse {el:.2e}")
