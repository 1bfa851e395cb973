"""moe_router_topk_noalloc: the router gemv + top-k for callers that cannot
allocate device memory (a runtime whose caching allocator owns all device
memory, a fixed up-front memory plan, or a latency-critical path where an
allocation could synchronise the device).  It keeps its scratch in a fixed
array inside the library instead of a handle's workspace.

Checked through the C ABI against the ids and weights that the allocating
entry point (moe_layer_forward_ex) returns for the same inputs, on two calls in
a row, with the parity tolerance of the other GPU tests.  This file is
collected last so that a failure here leaves every other test already run; it
passes alone in a fresh process as well as after the others.
"""
import numpy as np
import pytest

import moe_inputs as mi
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


def _device(a):
    if a is None:
        return None
    return gu.to_torch_x(a, "bf16") if a.dtype == np.uint16 else torch.from_numpy(
        np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("name,Ts", [("tiny", (4, 16)), ("latent", (1, 16, 64))])
def test_noalloc_routing_matches_layer_forward(name, Ts):
    import quantized_moe_decode_gemv_gb300 as pkg
    lay = gu.cached_layer(name)
    sp = lay.spec
    h = gu.build_layer(lay, max(Ts))
    try:
        router_w = _device(lay.router_w)
        bias = _device(lay.router_bias)
        for T in Ts:
            # two calls in a row, on different inputs, share the one scratch array
            for call in range(2):
                x, _ = gu.margin_x(lay, T, seed=300 + 10 * T + call)
                xt = gu.to_torch_x(x, sp.act_dtype)
                _, ids_ref, w_ref, _ = h.forward_ex(xt)
                ids = torch.full((T, sp.top_k), -1, dtype=torch.int32, device="cuda")
                w = torch.zeros((T, sp.top_k), dtype=torch.float32, device="cuda")
                stream = torch.cuda.current_stream().cuda_stream
                pkg.moe_router_topk_noalloc(xt, T, sp.hidden, sp.act_dtype, router_w,
                                            sp.router_dtype, bias, sp.n_experts, sp.top_k,
                                            sp.router, sp.renormalize, sp.routed_scale, ids, w,
                                            stream)
                torch.cuda.synchronize()
                assert np.array_equal(ids.cpu().numpy(), ids_ref.cpu().numpy()), (name, T, call)
                np.testing.assert_allclose(w.cpu().numpy(), w_ref.cpu().numpy(),
                                           rtol=gu.W_RTOL, atol=gu.W_ATOL)
    finally:
        h.close()


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import quantized_moe_decode_gemv_gb300 as pkg
    T = 65
    x = torch.zeros((T, 512), dtype=torch.bfloat16, device="cuda")
    wr = torch.zeros((16, 512), dtype=torch.bfloat16, device="cuda")
    ids = torch.empty((T, 2), dtype=torch.int32, device="cuda")
    w = torch.empty((T, 2), dtype=torch.float32, device="cuda")
    with pytest.raises(pkg.MoEError, match="UNSUPPORTED"):
        pkg.moe_router_topk_noalloc(x, T, 512, "bf16", wr, "bf16", None, 16, 2, "softmax", True,
                                    1.0, ids, w)
    with pytest.raises(pkg.MoEError, match="UNSUPPORTED"):
        pkg.moe_router_topk_noalloc(x, 4, 512, "bf16", wr, "bf16", None, 2048, 2, "softmax",
                                    True, 1.0, ids, w)
    with pytest.raises(pkg.MoEError, match="TOPK_GT_E"):
        pkg.moe_router_topk_noalloc(x, 4, 512, "bf16", wr, "bf16", None, 16, 17, "softmax",
                                    True, 1.0, ids, w)
