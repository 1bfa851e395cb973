"""moe_router_topk_noalloc: the router gemv + top-k for callers that cannot
allocate device memory (a runtime whose caching allocator owns all device
memory, a fixed up-front memory plan, or a latency-critical path where an
allocation could synchronise the device).  It keeps its scratch in a fixed
array inside the library instead of a handle's workspace.

Checked through the C ABI, on two calls in a row that share the one scratch
array: against the ids and weights that the allocating entry point
(moe_layer_forward_ex) returns for the same inputs, and against the fp64
oracle's routing of the same rows, with the routing tolerance of the other GPU
tests.  This file is collected last so that a failure here leaves every other
test already run; it passes alone in a fresh process as well as after the
others.
"""
import numpy as np
import pytest

import moe_inputs as mi
import oracle
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


def _oracle_routing(lay, x):
    """ids [T, k] and weights [T, k] of the fp64 oracle, row by row."""
    sp = lay.spec
    Wr = oracle.widen(lay.router_w, sp.router_dtype)
    bias = None if lay.router_bias is None else lay.router_bias.astype(np.float64)
    xs = oracle.widen(x, sp.act_dtype)
    ids, w = [], []
    for t in range(xs.shape[0]):
        i, ww = oracle.route(oracle.router_logits(xs[t], Wr), sp, bias)
        ids.append(i)
        w.append(ww)
    return np.array(ids), np.array(w)


def _noalloc(lay, xt, T, router_w, bias, key_status=None):
    import quantized_moe_decode_gemv_gb300 as pkg
    sp = lay.spec
    ids = torch.full((T, sp.top_k), -1, dtype=torch.int32, device="cuda")
    w = torch.zeros((T, sp.top_k), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    pkg.moe_router_topk_noalloc(xt, T, sp.hidden, sp.act_dtype, router_w, sp.router_dtype, bias,
                                sp.n_experts, sp.top_k, sp.router, sp.renormalize,
                                sp.routed_scale, ids, w, stream, key_status=key_status)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("name,Ts", [("tiny", (4, 16)), ("latent", (1, 16, 64))])
def test_noalloc_routing_matches_layer_forward_and_oracle(name, Ts):
    lay = gu.cached_layer(name)
    sp = lay.spec
    h = gu.build_layer(lay, max(Ts))
    try:
        router_w = _device(lay.router_w)
        bias = _device(lay.router_bias)
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        for T in Ts:
            # two calls in a row, on different inputs, share the one scratch array
            for call in range(2):
                x, _ = gu.margin_x(lay, T, seed=300 + 10 * T + call)
                xt = gu.to_torch_x(x, sp.act_dtype)
                _, ids_ref, w_ref, _ = h.forward_ex(xt)
                ids, w = _noalloc(lay, xt, T, router_w, bias, key_status=status)
                assert np.array_equal(ids, ids_ref.cpu().numpy()), (name, T, call)
                np.testing.assert_allclose(w, w_ref.cpu().numpy(), rtol=gu.W_RTOL, atol=gu.W_ATOL)
                ora_ids, ora_w = _oracle_routing(lay, x)
                assert np.array_equal(ids, ora_ids), (name, T, call)
                np.testing.assert_allclose(w, ora_w, rtol=gu.W_RTOL, atol=gu.W_ATOL)
                assert int(status.item()) == 0
    finally:
        h.close()


def test_noalloc_reports_non_finite_keys():
    """NaN selection biases: those experts rank last (as in the oracle) and the
    caller's status word says so; the next call on finite keys clears it."""
    spec = mi.LayerSpec(name="nan_bias", hidden=512, n_experts=16, top_k=3, expert_ffn=128,
                        latent=0, group_size=64, shared_ffn=0, act="relu2", router="sigmoid",
                        routed_scale=1.0, router_bias=True, weight_std=0.05)
    lay = mi.make_layer(spec, 5)
    clean = lay.router_bias.copy()
    lay.router_bias[[2, 7, 11]] = np.nan
    T = 4
    x, _ = gu.margin_x(lay, T, seed=81)
    xt = gu.to_torch_x(x, "bf16")
    router_w = _device(lay.router_w)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    ids, w = _noalloc(lay, xt, T, router_w, _device(lay.router_bias), key_status=status)
    ora_ids, ora_w = _oracle_routing(lay, x)
    assert np.array_equal(ids, ora_ids)
    np.testing.assert_allclose(w, ora_w, rtol=gu.W_RTOL, atol=gu.W_ATOL)
    assert not np.isin(ids, [2, 7, 11]).any()
    assert int(status.item()) == 1
    lay.router_bias[:] = clean
    _noalloc(lay, xt, T, router_w, _device(lay.router_bias), key_status=status)
    assert int(status.item()) == 0


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
