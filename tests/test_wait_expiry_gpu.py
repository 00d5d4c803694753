"""The bounded device-side waits run out, on purpose, through the test hook
pa_debug_wait_expiry: every wait helper the kernels use must return after its
limit, set PA_DEVICE_WAIT_TIMEOUT in the scratch header, and leave the context
usable; a helper that finds the bit already set (another CTA's wait expired)
must give up at once.  Nothing arrives on the awaited mbarrier and nothing
else is in flight, so the only way out is the limit on %globaltimer."""
import numpy as np
import pytest

from paged_kv_gqa_12_gb300 import workloads as wl
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu

LIMIT_NS = 2_000_000   # 2 ms


@pytest.fixture(scope="module")
def pb():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_gqa_12_gb300 import binding
    binding.load()
    return binding


def _scratch(pb):
    import torch
    buf = torch.empty(pb.SCRATCH_HEADER_BYTES + 256, dtype=torch.uint8, device="cuda")
    off = (-buf.data_ptr()) % 256
    s = buf[off:off + pb.SCRATCH_HEADER_BYTES]
    pb.scratch_init(s)
    return s


def _result(s):
    import torch
    torch.cuda.synchronize()
    return s[64:80].cpu().numpy().view(np.int64)


@pytest.mark.parametrize("which", [0, 1, 2])
def test_wait_expires_and_reports(pb, which):
    s = _scratch(pb)
    pb.debug_wait_expiry(s, which, LIMIT_NS)
    saw, waited = _result(s)
    assert saw == 0
    assert LIMIT_NS <= waited < 1_000_000_000, waited
    assert pb.check(s) == pb.DEVICE_WAIT_TIMEOUT
    assert pb.check(s) == 0                 # pa_check cleared the header


@pytest.mark.parametrize("which", [3, 4])
def test_wait_gives_up_after_another_expiry(pb, which):
    s = _scratch(pb)
    limit = 50_000_000                       # 50 ms: far longer than giving up should take
    pb.debug_wait_expiry(s, which, limit)
    saw, waited = _result(s)
    assert saw == 0
    assert waited < limit // 5, waited
    assert pb.check(s) == pb.DEVICE_WAIT_TIMEOUT


def test_context_usable_after_expiry(pb):
    # an attention call on the same stream right after an expired wait runs
    # normally and matches the oracle
    import oracle
    s = _scratch(pb)
    pb.debug_wait_expiry(s, 1, LIMIT_NS)
    assert pb.check(s) == pb.DEVICE_WAIT_TIMEOUT
    p = wl.build_problem("decode", num_q_heads=8, num_kv_heads=2, head_dim=64, page_size=16,
                         seq_lens=[1, 37, 300, 129], seed=7, window=100, sinks=True)
    ref_o, ref_l = oracle.attention(p)
    out, lse = gh.run(p, num_splits=4)
    gh.assert_parity(out, lse, ref_o, ref_l, what="decode after an expired wait")


def test_rejects_bad_arguments(pb):
    s = _scratch(pb)
    for which, limit in ((5, LIMIT_NS), (-1, LIMIT_NS), (0, 10), (0, 10**9)):
        with pytest.raises(pb.PaError) as ei:
            pb.debug_wait_expiry(s, which, limit)
        assert ei.value.status == pb.PA_ERR_INVALID_ARG
