"""The one-launch decode layer (moe_decode_layer) against the oracle.

The call runs route, admission/permutation, the grouped SwiGLU and the combine
of [M6.6] 0x03-0x04 as one kernel for at most 64 routes.  Every output is
compared with the oracle: routing ids, counts, offsets, both maps and drops bit
for bit, the permuted rows as bit copies, gates to the gate tolerance, H, y and
the fp32 output to the float bar.  The workspace counters must be zero again
after every call, and a replayed graph must give the eager call's bits.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from moe_check import (assert_float_parity, assert_gates, bits, host, oracle_expert_rows,
                       oracle_route, weights_fetcher)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    from grouped_expert_gemm_gb300 import build
    build.build()


@pytest.fixture(scope="module")
def decode_weights():
    return workloads.make_expert_weights(workloads.decode(128), DEV)


def make_layer(w, weights, capacity=-1, sel_bias=None, decode_path="fused"):
    import grouped_expert_gemm_gb300 as g
    score = g.MOE_SCORE_SOFTMAX if w.score_fn == "softmax" else g.MOE_SCORE_SIGMOID_GROUP
    wg, wu, wd = weights
    return g.MoELayer(w.T, w.d, w.E, w.k, w.I, wg, wu, wd, capacity=capacity, score_fn=score,
                      n_group=w.n_group, topk_group=w.topk_group, route_scale=w.route_scale,
                      sel_bias=sel_bias, decode_path=decode_path, device=DEV)


def check_against_oracle(w, layer, logits, sel_bias, x, weights, capacity, valid=None):
    """Every output of one decode call against the oracle on the live tokens."""
    T, k = w.T, w.k
    live = T if valid is None else valid
    assert int(layer.dev_status.item()) == 0
    ids_all = host(layer.topk_ids)
    if live > 0:
        wl = workloads.scaled(w, T=live)
        ids, gates = oracle_route(wl, logits[:live], sel_bias)
        assert np.array_equal(ids_all[:live], ids)
        assert_gates(host(layer.gates)[:live], gates)
    else:
        ids = np.zeros((0, k), np.int32)
        gates = np.zeros((0, k))
    perm = oracle.permute(ids, w.E, capacity)
    acc = int(perm["offsets"][-1])
    assert np.array_equal(host(layer.counts), perm["counts"])
    assert np.array_equal(host(layer.offsets), perm["offsets"])
    assert int(layer.n_dropped.item()) == perm["n_dropped"]
    assert np.array_equal(host(layer.row_to_route)[:acc], perm["row_to_route"])
    r2r = host(layer.route_to_row)
    assert np.array_equal(r2r[: live * k], perm["route_to_row"])
    # padding slots of a bucket: no identity, no gate, no row, zero output
    assert np.all(ids_all[live:] == -1)
    assert np.all(host(layer.gates)[live:] == 0)
    assert np.all(r2r[live * k: T * k] == -1)
    assert np.all(host(layer.out)[live:] == 0)
    xb = bits(x)
    if acc == 0:
        return
    rows = np.arange(acc)
    tok = perm["row_to_route"] // k
    assert np.array_equal(bits(layer.x_perm[:acc]), xb[tok])
    seg = np.searchsorted(perm["offsets"], rows, side="right") - 1
    h_ref, y_ref = oracle_expert_rows(rows, seg, xb[tok], weights_fetcher(*weights))
    assert_float_parity(oracle.bf16_to_f64(bits(layer.H[:acc])), h_ref, "decode H")
    assert_float_parity(oracle.bf16_to_f64(bits(layer.y[:acc])), y_ref, "decode y")
    y_rows = np.zeros((max(acc, 1), w.d))
    y_rows[:acc] = oracle.bf16_to_f64(bits(layer.y[:acc]))
    # the combine on the device's own y: fp32 slot-order sums, compared to fp64
    ref = oracle.combine(y_rows, perm["route_to_row"], gates, live, k)
    assert_float_parity(host(layer.out)[:live], ref, "decode combined output")
    # and on the oracle's y
    y_o = np.zeros((max(acc, 1), w.d))
    y_o[:acc] = y_ref
    assert_float_parity(host(layer.out)[:live],
                        oracle.combine(y_o, perm["route_to_row"], gates, live, k),
                        "decode output against oracle y")


def counters_zero(layer):
    """The workspace starts with the call's counters (claims, finished CTAs, 64 row-group
    H counts, one y count per 64-column block of d, one count per row group and
    64-column block of I); they must be zero again after the call."""
    words = 2 + 64 + layer.d // 64 + 64 * (layer.I // 64)
    return int(layer.decode_ws[: 4 * words].view(torch.int32).abs().sum().item()) == 0


@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 8])
def test_decode_layer_matches_the_oracle(T, decode_weights):
    w = workloads.decode(T)
    logits, _ = workloads.make_router_inputs(w, DEV)
    x = workloads.make_activations(w, DEV)
    layer = make_layer(w, decode_weights)
    assert layer.fused
    layer.forward(logits, x)
    torch.cuda.synchronize()
    check_against_oracle(w, layer, logits, None, x, decode_weights, -1)
    assert counters_zero(layer)


def test_decode_layer_equals_the_separate_calls(decode_weights):
    """The same step through the per-stage calls: identical integers and copied rows;
    H, y and the output within the float bar of each other."""
    w = workloads.decode(8)
    logits, _ = workloads.make_router_inputs(w, DEV)
    x = workloads.make_activations(w, DEV)
    fused = make_layer(w, decode_weights)
    sep = make_layer(w, decode_weights, decode_path="separate")
    fused.forward(logits, x)
    sep.forward(logits, x)
    torch.cuda.synchronize()
    for name in ("topk_ids", "counts", "offsets", "n_dropped"):
        assert torch.equal(getattr(fused, name), getattr(sep, name)), name
    assert torch.equal(fused.gates, sep.gates)
    R, acc = w.R, int(sep.offsets[-1].item())
    assert torch.equal(fused.route_to_row[:R], sep.route_to_row[:R])
    assert torch.equal(fused.row_to_route[:acc], sep.row_to_route[:acc])
    assert torch.equal(fused.x_perm[:acc].view(torch.int16), sep.x_perm[:acc].view(torch.int16))
    assert_float_parity(host(fused.H[:acc].float()), host(sep.H[:acc].float()), "H fused/separate")
    assert_float_parity(host(fused.y[:acc].float()), host(sep.y[:acc].float()), "y fused/separate")
    assert_float_parity(host(fused.out), host(sep.out), "out fused/separate")


@pytest.mark.parametrize("case", ["capacity_drops", "grouped", "wide_E", "ragged_slices"])
def test_decode_layer_shapes(case):
    """Capacity with drops in route-id order; the group-limited sigmoid router; 512
    experts with k = 16; d and I that leave a short last row slice."""
    sel_bias = None
    cap = -1
    if case == "capacity_drops":
        w = workloads.scaled(workloads.tiny(), T=16, E=8, k=4, d=128, I=128)
        cap = 3
    elif case == "grouped":
        w = workloads.scaled(workloads.v3(), T=4, E=64, k=6, d=256, I=128, n_group=4,
                             topk_group=2, shared_I=0)
    elif case == "wide_E":
        w = workloads.scaled(workloads.tiny(), T=4, E=512, k=16, d=1024, I=192)
    else:
        w = workloads.scaled(workloads.tiny(), T=2, E=16, k=4, d=320, I=320)
    logits, sel_bias = workloads.make_router_inputs(w, DEV)
    x = workloads.make_activations(w, DEV)
    weights = workloads.make_expert_weights(w, DEV)
    layer = make_layer(w, weights, capacity=cap, sel_bias=sel_bias)
    assert layer.fused
    layer.forward(logits, x)
    torch.cuda.synchronize()
    check_against_oracle(w, layer, logits, sel_bias, x, weights, cap)
    if case == "capacity_drops":
        assert int(layer.n_dropped.item()) > 0
    assert counters_zero(layer)


@pytest.mark.parametrize("valid", [0, 1, 3, 4])
def test_decode_layer_with_a_valid_count(valid, decode_weights):
    """A 4-slot bucket with `valid` live tokens: the live tokens get the oracle's
    results, the padding slots stay masked with zero output."""
    w = workloads.decode(4)
    logits, _ = workloads.make_router_inputs(w, DEV)
    x = workloads.make_activations(w, DEV)
    layer = make_layer(w, decode_weights)
    vt = torch.tensor([valid], dtype=torch.int32, device=DEV)
    layer.out.fill_(7.0)
    layer.decode_layer(logits, x, valid_tokens=vt)
    torch.cuda.synchronize()
    check_against_oracle(w, layer, logits, None, x, decode_weights, -1, valid=valid)
    assert counters_zero(layer)


def test_decode_layer_replays_from_a_graph(decode_weights):
    """Several replays of one captured call on changing inputs: each gives the eager
    call's bits, and the counters are zero after every replay."""
    w = workloads.decode(2)
    layer = make_layer(w, decode_weights)
    ref_layer = make_layer(w, decode_weights)
    logits = torch.empty((w.T, w.E), device=DEV)
    x = torch.empty((w.T, w.d), dtype=torch.bfloat16, device=DEV)
    stream = torch.cuda.Stream(DEV)
    with torch.cuda.stream(stream):
        layer.forward(logits.normal_(), x.normal_())
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        layer.forward(logits, x)
    for seed in range(3):
        gen = torch.Generator(device=DEV).manual_seed(seed)
        logits.copy_(torch.randn((w.T, w.E), generator=gen, device=DEV))
        x.copy_(torch.randn((w.T, w.d), generator=gen, device=DEV).to(torch.bfloat16))
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            graph.replay()
        stream.synchronize()
        ref_layer.forward(logits, x)
        torch.cuda.synchronize()
        assert torch.equal(layer.out, ref_layer.out)
        assert torch.equal(layer.topk_ids, ref_layer.topk_ids)
        assert counters_zero(layer)
