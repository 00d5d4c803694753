"""Seeded random parity cases: shapes and options drawn together (group size,
head_dim, page size, window, soft-cap, sinks, e4m3 cache with per-tensor or
per-request scales, split counts, ragged lengths with empty requests) for
decode, verify and extend, each against the oracle."""
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


def _draw(seed, mode):
    rng = np.random.default_rng(seed)
    D = int(rng.choice([64, 128, 256]))
    ps = int(rng.choice([16, 32, 64]))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.choice([1, 2, 3, 4, 8, 16] + ([20, 32] if mode != "verify" else [])))
    if mode == "verify":
        q_len = int(rng.integers(1, max(2, 16 // G + 1)))
        while q_len * G > 16:
            q_len -= 1
    B = int(rng.integers(1, 7))
    opts = {}
    if rng.random() < 0.4:
        opts["window"] = int(rng.integers(1, 700))
    if rng.random() < 0.3:
        opts["soft_cap"] = float(rng.uniform(3.0, 30.0))
    if rng.random() < 0.4:
        opts["sinks"] = True
    kv = "fp8_e4m3" if rng.random() < 0.4 else "bf16"
    if kv == "fp8_e4m3":
        if rng.random() < 0.5:
            opts["k_scales"] = np.exp(rng.uniform(np.log(0.01), np.log(0.2), size=B)).astype(np.float32)
            opts["v_scales"] = np.exp(rng.uniform(np.log(0.01), np.log(0.2), size=B)).astype(np.float32)
        else:
            opts["k_scale"], opts["v_scale"] = 0.05, 0.07
    common = dict(num_q_heads=G * Hkv, num_kv_heads=Hkv, head_dim=D, page_size=ps, kv_dtype=kv, seed=seed, **opts)
    if mode == "decode":
        lens = rng.integers(0, 1500, size=B)
        lens[rng.random(B) < 0.15] = 0
        return wl.build_problem("decode", seq_lens=lens, **common), {}
    if mode == "verify":
        ctx = rng.integers(0, 1500, size=B)
        ql = np.full(B, q_len)
        return wl.build_problem("extend", seq_lens=ctx + ql, query_lens=ql, **common), {"verify": True}
    ctx = rng.integers(0, 1200, size=B)
    ql = rng.integers(0, 300, size=B)
    ql[0] = max(ql[0], 1)
    return wl.build_problem("extend", seq_lens=ctx + ql, query_lens=ql, **common), {}


@pytest.mark.parametrize("seed", range(12))
@pytest.mark.parametrize("mode", ["decode", "verify", "extend"])
def test_random_case(mode, seed):
    p, kw = _draw(7000 + 97 * seed + len(mode), mode)
    ref_o, ref_l = oracle.attention(p)
    if mode == "decode":
        # planner, two and eleven splits (more than the eight the merge folds
        # at once), and a capacity-only plan with room for more requests
        for ns in (0, 2, 11):
            out, lse = gh.run(p, num_splits=ns)
            gh.assert_parity(out, lse, ref_o, ref_l, what=f"{mode} seed {seed} splits {ns}")
        plan = gh.make_plan(p, host_lens=False, max_batch=p.batch + 3)
        out, lse = gh.run(p, plan=plan)
        gh.assert_parity(out, lse, ref_o, ref_l, what=f"{mode} seed {seed} capacity plan")
    else:
        out, lse = gh.run(p, **kw)
        gh.assert_parity(out, lse, ref_o, ref_l, what=f"{mode} seed {seed}")
