"""GPU parity of the calls beyond the forward path: the backward of the
transpose (combine backward, token-gradient unpermute) and the load telemetry /
bias controller step, against the CPU oracle."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import workloads
from moe_check import assert_float_parity, bits, host

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    from grouped_expert_gemm_gb300 import build
    build.build()


def G():
    import grouped_expert_gemm_gb300 as g
    return g


def _case(T, k, d, rows, drop_frac, seed):
    rng = np.random.default_rng(seed)
    r2r = rng.permutation(rows)[: T * k].astype(np.int32)
    r2r[rng.random(T * k) < drop_frac] = -1
    gates = rng.uniform(0, 1, T * k).astype(np.float32)
    gen = torch.Generator(device=DEV).manual_seed(seed)
    y = torch.randn((rows, d), generator=gen, device=DEV).to(torch.bfloat16)
    dout = torch.randn((T, d), generator=gen, device=DEV, dtype=torch.float32)
    return r2r, gates, y, dout


@pytest.mark.parametrize("T,k,d,rows,drop", [(64, 2, 64, 200, 0.0), (33, 8, 2048, 300, 0.2),
                                              (100, 16, 1032, 1700, 0.1), (7, 1, 8, 9, 0.3),
                                              (256, 4, 4096, 1100, 0.05)])
def test_combine_backward_parity(T, k, d, rows, drop):
    g = G()
    r2r, gates, y, dout = _case(T, k, d, rows, drop, seed=T + k)
    sentinel = torch.full((rows, d), 3.0, dtype=torch.bfloat16, device=DEV)
    dy = sentinel.clone()
    dg = torch.full((T * k,), 9.0, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    g.moe_combine_backward(T, k, d, dout, y, rows, torch.from_numpy(r2r).to(DEV),
                           torch.from_numpy(gates).to(DEV), dy, dg, st)
    torch.cuda.synchronize()
    assert int(host(st)[0]) == 0
    ref_dy, ref_dg = oracle.combine_backward(host(dout).astype(np.float64),
                                             oracle.bf16_to_f64(bits(y)), r2r, gates, T, k)
    acc = r2r[r2r >= 0]
    assert_float_parity(oracle.bf16_to_f64(bits(dy)[acc]), ref_dy[acc], "dy")
    # rows of no accepted route are never written
    untouched = np.setdiff1d(np.arange(rows), acc)
    assert np.array_equal(bits(dy)[untouched], bits(sentinel)[untouched])
    assert_float_parity(host(dg), ref_dg.reshape(-1), "dgates")
    np.testing.assert_allclose(host(dg), ref_dg.reshape(-1), rtol=1e-4,
                               atol=1e-4 * np.abs(ref_dg).max())
    assert np.all(host(dg)[r2r < 0] == 0)


@pytest.mark.parametrize("accumulate", [0, 1])
def test_unpermute_grad_parity(accumulate):
    g = G()
    T, k, d, rows = 129, 8, 2048, 1100
    r2r, _, dxp, _ = _case(T, k, d, rows, 0.1, seed=5)
    init = torch.randn((T, d), device=DEV, dtype=torch.float32)
    dx = init.clone()
    g.moe_unpermute_grad(T, k, d, dxp, rows, torch.from_numpy(r2r).to(DEV), dx, accumulate)
    torch.cuda.synchronize()
    ref = oracle.unpermute_grad(oracle.bf16_to_f64(bits(dxp)), r2r, T, k)
    if accumulate:
        ref = ref + host(init)
    assert_float_parity(host(dx), ref, "dx")
    np.testing.assert_allclose(host(dx), ref, rtol=1e-5, atol=1e-5)


def test_backward_of_the_layer_transpose():
    """Forward through the library, then the transpose backward on its own maps."""
    import grouped_expert_gemm_gb300 as g
    w = workloads.scaled(workloads.v3(), T=96, d=256, I=256, shared_I=0)
    logits, sb = workloads.make_router_inputs(w, DEV)
    x = workloads.make_activations(w, DEV)
    wg, wu, wd = workloads.make_expert_weights(w, DEV)
    cap = g.capacity_from_factor(w.capacity_factor, w.R, w.E)
    layer = g.MoELayer(w.T, w.d, w.E, w.k, w.I, wg, wu, wd, capacity=cap,
                       score_fn=g.MOE_SCORE_SIGMOID_GROUP, n_group=w.n_group,
                       topk_group=w.topk_group, route_scale=w.route_scale, sel_bias=sb, device=DEV)
    layer.forward(logits, x)
    dout = torch.randn((w.T, w.d), device=DEV, dtype=torch.float32)
    R = w.R
    dy = torch.zeros((R, w.d), dtype=torch.bfloat16, device=DEV)
    dg = torch.empty((R,), dtype=torch.float32, device=DEV)
    g.moe_combine_backward(w.T, w.k, w.d, dout, layer.y, R, layer.route_to_row, layer.gates, dy,
                           dg, layer.dev_status)
    dx = torch.empty((w.T, w.d), dtype=torch.float32, device=DEV)
    g.moe_unpermute_grad(w.T, w.k, w.d, dy, R, layer.route_to_row, dx, 0, layer.dev_status)
    torch.cuda.synchronize()
    assert int(layer.dev_status.item()) == 0
    r2r = host(layer.route_to_row)[:R]
    acc = int(host(layer.offsets)[-1])
    ref_dy, ref_dg = oracle.combine_backward(host(dout).astype(np.float64),
                                             oracle.bf16_to_f64(bits(layer.y)), r2r,
                                             host(layer.gates).reshape(-1), w.T, w.k)
    assert_float_parity(oracle.bf16_to_f64(bits(dy)[:acc]), ref_dy[:acc], "dy")
    assert_float_parity(host(dg), ref_dg.reshape(-1), "dgates")
    ref_dx = oracle.unpermute_grad(oracle.bf16_to_f64(bits(dy)), r2r, w.T, w.k)
    np.testing.assert_allclose(host(dx), ref_dx, rtol=1e-5, atol=1e-5)


def _stats(counts):
    g = G()
    c = torch.tensor(counts, dtype=torch.int32, device=DEV)
    out = torch.empty(5, dtype=torch.float64, device=DEV)
    g.moe_load_stats(len(counts), c, out)
    torch.cuda.synchronize()
    return host(out)


def test_load_stats_parity():
    rng = np.random.default_rng(7)
    cases = [rng.integers(0, 50, 384).tolist(), [0] * 10 + [5], [3], [0, 0, 0],
             rng.poisson(3, 4000).tolist()]
    with open(os.path.join(os.path.dirname(__file__), "golden", "m62_load_and_controller.json")) as f:
        fx = json.load(f)
    cases += [v[0] for v in fx["cv2_by_axis"].values()] + [fx["maxvio_toy"]["counts"]]
    for c in cases:
        ref = oracle.load_stats(c)
        got = _stats(c)
        np.testing.assert_allclose(got, [ref["cv2"], ref["rho_max"], ref["h_norm"], ref["e_eff"],
                                         ref["max_vio"]], rtol=1e-12, atol=1e-14)
    for counts, cv2 in fx["cv2_by_axis"].values():
        assert abs(_stats(counts)[0] - cv2) < 1e-12


@pytest.mark.parametrize("rule", [0, 1])
def test_bias_update_bit_exact(rule):
    g = G()
    rng = np.random.default_rng(8 + rule)
    E = 384
    counts = rng.integers(0, 40, E).astype(np.int32)
    b0 = (rng.standard_normal(E) * 0.1).astype(np.float32)
    bias = torch.from_numpy(b0.copy()).to(DEV)
    u = 1e-3 if rule == 0 else 3e-4
    g.moe_bias_update(E, torch.from_numpy(counts).to(DEV), bias, u, rule)
    torch.cuda.synchronize()
    ref = oracle.bias_update(b0, counts, u, "sign" if rule == 0 else "proportional")
    assert np.array_equal(host(bias).view(np.uint32), ref.view(np.uint32))


def test_bias_update_page_fixture():
    g = G()
    with open(os.path.join(os.path.dirname(__file__), "golden", "m62_load_and_controller.json")) as f:
        fx = json.load(f)["controller"]
    c = np.array(fx["counts"], np.int32)
    bias = torch.zeros(c.size, dtype=torch.float32, device=DEV)
    g.moe_bias_update(c.size, torch.from_numpy(c).to(DEV), bias, fx["gamma"], g.MOE_BIAS_SIGN)
    torch.cuda.synchronize()
    b = host(bias)
    assert all(b[e] == np.float32(-0.001) for e in fx["decrease"])
    assert all(b[e] == np.float32(0.001) for e in fx["increase_zero_load"])


@pytest.mark.parametrize("rule", [0, 1])
def test_layer_bias_step_on_v3_routing(rule):
    """MoELayer.bias_step after a V3-routed batch: the demand of that batch (before the
    capacity of 1.0) and the controller step on the layer's selection bias, bit-exact."""
    import grouped_expert_gemm_gb300 as g
    w = workloads.scaled(workloads.v3(), T=512, d=256, I=256, shared_I=0)
    logits, sel_bias = workloads.make_router_inputs(w, DEV)
    wg, wu, wd = workloads.make_expert_weights(w, DEV)
    cap = g.capacity_from_factor(w.capacity_factor, w.R, w.E)
    layer = g.MoELayer(w.T, w.d, w.E, w.k, w.I, wg, wu, wd, capacity=cap,
                       score_fn=g.MOE_SCORE_SIGMOID_GROUP, n_group=w.n_group,
                       topk_group=w.topk_group, route_scale=w.route_scale, sel_bias=sel_bias,
                       device=DEV)
    b0 = host(sel_bias).copy()
    layer.route(logits)
    u = 1e-3 if rule == 0 else 2e-4
    layer.bias_step(u, rule)
    torch.cuda.synchronize()
    ids = host(layer.topk_ids)
    demand = oracle.expert_demand(ids, w.E)
    assert host(layer.demand).tolist() == demand.tolist()
    assert demand.max() > cap  # the capped counts would hide the overload
    ref = oracle.bias_update(b0, demand, u, "sign" if rule == 0 else "proportional")
    assert np.array_equal(host(layer.sel_bias).view(np.uint32), ref.view(np.uint32))
