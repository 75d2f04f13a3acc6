"""Failure detection on the device without a fault: a bounded wait on an
mbarrier that nothing completes gives up after its limit, reports
DS_VIT_ETIMEOUT through the status word, and the context stays usable (an
op launched afterwards still matches the oracle)."""
import pytest

import oracle as O
from gpu_util import dev, host, rand_bits, rel_err

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def dv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import vit_vision_encoder_gb300
    return vit_vision_encoder_gb300


@pytest.mark.parametrize("limit_us", [200, 5000])
def test_bounded_wait_times_out(dv, limit_us):
    status, waited_ns = dv.selftest_wait_timeout(limit_us)
    assert status == dv.ETIMEOUT
    assert waited_ns >= limit_us * 1000
    assert waited_ns < limit_us * 1000 + 50_000_000     # gave up, did not keep waiting


def test_context_usable_after_timeout(dv):
    status, _ = dv.selftest_wait_timeout(1000)
    assert status == dv.ETIMEOUT
    M = 300
    x = rand_bits((M, 1024), 90)
    g = rand_bits(1024, 91, 0.5)
    b = rand_bits(1024, 92, 0.5)
    y = dv.op_layernorm(dev(x, torch), dev(g, torch), dev(b, torch))
    torch.cuda.synchronize()
    ref = O.round_bf16(O.layer_norm(O.bits_to_f32(x), O.bits_to_f32(g), O.bits_to_f32(b), 1e-6))
    got = host(y)
    assert rel_err(got, ref).max() <= 8e-3
    assert (got == ref).mean() > 0.99
