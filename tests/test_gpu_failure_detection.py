"""Failure detection without a GPU fault: a bounded device-side wait that runs
out is recorded in the handle's status word, the launch still completes, the
host reads MOE_ERR_TIMEOUT, and the next forward is exact again.

The dense pass's routing CTA is made to wait for one router CTA more than
exist (MOE_DEBUG_STALL=1, read by the launcher at every launch), so its bounded
wait runs out.  No kernel traps, faults or hangs: every wait in the library is
bounded, and a CTA whose wait ran out still completes its work (the routing runs
on the logits as they stand), so the launch completes and the next forward is
exact.
"""
import pytest

from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    yield
    torch.cuda.synchronize()


def test_routing_wait_timeout_is_reported_and_recovers(monkeypatch):
    import quantized_moe_decode_gemv_gb300 as pkg
    lay = gu.cached_layer("tiny")
    h = gu.build_layer(lay, 4)
    try:
        h.set_path("gemv")
        x, _ = gu.margin_x(lay, 4, seed=124)
        xt = gu.to_torch_x(x, lay.spec.act_dtype)
        assert h.device_status() == 0
        monkeypatch.setenv("MOE_DEBUG_STALL", "1")
        h.forward(xt)
        torch.cuda.synchronize()
        assert pkg._capi.STATUS_NAMES[h.device_status()] == "MOE_ERR_TIMEOUT"
        monkeypatch.delenv("MOE_DEBUG_STALL")
        got = gu.run_layer(h, x, lay.spec.act_dtype)
        gu.check_parity(got, gu.ora_forward(lay, x), what="after a recorded routing timeout")
        assert h.device_status() == 0
    finally:
        h.close()
