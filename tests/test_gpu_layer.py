"""End-to-end parity of the MoE layer (the launch configuration the benchmark
times) against the CPU oracle.

Small workloads are checked in full.  The full-size workloads are run whole on
the GPU; routing, admission, permutation, pool headers and maps are compared in
full (bit-exact), payload copies and float outputs on a seeded sample of tokens
and rows that the oracle computes one by one.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from moe_check import (assert_every_tile_reached, assert_float_parity, assert_gates, bits, host,
                       oracle_capacity, oracle_expert_rows, oracle_route, oracle_token_outputs,
                       stratified_rows, weights_fetcher, weights_fetcher_uncached)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    from grouped_expert_gemm_gb300 import build
    build.build()


def make_layer(w, wg, wu, wd, sel_bias=None, shared=None, payload="bf16", gather=False,
               fp8_loader="auto"):
    import grouped_expert_gemm_gb300 as g
    cap = -1 if w.capacity_factor is None else g.capacity_from_factor(w.capacity_factor, w.R, w.E)
    score = g.MOE_SCORE_SOFTMAX if w.score_fn == "softmax" else g.MOE_SCORE_SIGMOID_GROUP
    return g.MoELayer(w.T, w.d, w.E, w.k, w.I, wg, wu, wd, capacity=cap, score_fn=score,
                      n_group=w.n_group, topk_group=w.topk_group, route_scale=w.route_scale,
                      sel_bias=sel_bias, shared_weights=shared, payload=payload, gather=gather,
                      fp8_loader=fp8_loader, device=DEV)


SCALE_GROUP = {"fp8_row": 0, "fp8_block128": 128}


def run_and_check(w, sample_tokens=None, sample_rows=64, seed=0, weights=None, payload="bf16",
                  gather=False, fp8_loader="auto", every_tile=False):
    """The layer on workload `w` against the oracle.  With every_tile, H and y are also
    checked on rows that reach every 128-row m-tile of every expert segment."""
    logits, sel_bias = workloads.make_router_inputs(w, DEV)
    x = workloads.make_activations(w, DEV)
    wg, wu, wd = weights if weights is not None else workloads.make_expert_weights(w, DEV)
    shared = workloads.make_shared_weights(w, DEV)
    layer = make_layer(w, wg, wu, wd, sel_bias, shared, payload, gather, fp8_loader)
    out = layer.forward(logits, x)
    torch.cuda.synchronize()
    assert int(layer.dev_status.item()) == 0

    # routing and admission: bit-exact in full
    ids, gates = oracle_route(w, logits, sel_bias)
    assert np.array_equal(host(layer.topk_ids), ids)
    assert_gates(host(layer.gates), gates)
    cap = oracle_capacity(w)
    perm = oracle.permute(ids, w.E, cap)
    assert np.array_equal(host(layer.counts), perm["counts"])
    assert np.array_equal(host(layer.offsets), perm["offsets"])
    acc = int(perm["offsets"][-1])
    assert np.array_equal(host(layer.row_to_route)[:acc], perm["row_to_route"])
    assert np.array_equal(host(layer.route_to_row)[: w.R], perm["route_to_row"])
    assert int(layer.n_dropped.item()) == perm["n_dropped"]

    xb = bits(x)
    rng = np.random.default_rng(seed)
    rows = np.arange(acc) if acc <= sample_rows else np.sort(rng.choice(acc, sample_rows, False))
    rows_dev = torch.from_numpy(rows).to(DEV)
    tok_of_row = perm["row_to_route"][rows] // w.k
    x_expert = xb  # the bf16 rows the experts see (token order)
    if payload == "bf16" and layer.gather:
        # no permuted copy: the gate/up pass gathers the rows (checked through H and y)
        assert not hasattr(layer, "x_perm")
    elif payload == "bf16":
        # permuted payload rows: bit copies
        assert np.array_equal(bits(layer.x_perm[rows_dev]), xb[tok_of_row])
    else:
        # E4M3 codes and scales of every token, bit-exact; permuted together
        grp = SCALE_GROUP[payload]
        q, sc = oracle.quantize_fp8(xb, grp)
        assert np.array_equal(host(layer.xq), q)
        assert np.array_equal(host(layer.xs).view(np.uint32), sc.view(np.uint32))
        assert np.array_equal(host(layer.xq_perm[rows_dev]), q[tok_of_row])
        assert np.array_equal(host(layer.xs_perm[rows_dev]).view(np.uint32),
                              sc[tok_of_row].view(np.uint32))
        x_expert = oracle.dequantize_fp8(q, sc, grp)
        if not layer.fused_fp8:  # dequantized once into bf16 rows before the gate/up pass
            assert np.array_equal(bits(layer.x_perm[rows_dev]), x_expert[tok_of_row])
    shared_x = xb

    tokens = np.arange(w.T) if sample_tokens is None else np.sort(
        rng.choice(w.T, min(sample_tokens, w.T), replace=False))
    shared_bits = None if shared is None else tuple(bits(s) for s in shared)
    ref_out, y_of_row = oracle_token_outputs(w, tokens, x_expert, ids, gates, perm,
                                             weights_fetcher(wg, wu, wd), shared_bits,
                                             shared_x_bits=shared_x)
    if y_of_row:
        yrows = np.array(sorted(y_of_row))
        got_y = oracle.bf16_to_f64(bits(layer.y[torch.from_numpy(yrows).to(DEV)]))
        assert_float_parity(got_y, np.stack([y_of_row[r] for r in yrows]), "expert rows y")
    got = host(out)[tokens]
    assert_float_parity(got, ref_out, "combined output")
    if every_tile:
        trows = stratified_rows(perm["offsets"][:-1], perm["counts"], rng)
        assert_every_tile_reached(trows, perm["offsets"][:-1], perm["counts"])
        seg = np.searchsorted(perm["offsets"], trows, side="right") - 1
        tok = perm["row_to_route"][trows] // w.k
        h_ref, y_ref = oracle_expert_rows(trows, seg, x_expert[tok],
                                          weights_fetcher_uncached(wg, wu, wd))
        idx = torch.from_numpy(trows).to(DEV)
        assert_float_parity(oracle.bf16_to_f64(bits(layer.H[idx])), h_ref, "H on every m-tile")
        assert_float_parity(oracle.bf16_to_f64(bits(layer.y[idx])), y_ref, "y on every m-tile")
    return layer, perm


def test_tiny_full():
    w = workloads.tiny()
    layer, perm = run_and_check(w, every_tile=True)
    assert oracle.capacity(1.25, 256, 2, 8) == layer.capacity == 80


@pytest.fixture(scope="module")
def decode_weights():
    return workloads.make_expert_weights(workloads.decode(128), DEV)


@pytest.mark.parametrize("T", [1, 2, 4, 8, 32, 128])  # 1, 4: narrow gate/up tiles; 1: narrow down
def test_decode_sweep_full(T, decode_weights):
    run_and_check(workloads.decode(T), weights=decode_weights, sample_rows=4096, every_tile=True)


@pytest.mark.parametrize("case", ["decode_hot8", "tiny_hot2_capacity", "prefill_hot2",
                                  "v3_hot_group"])
def test_degenerate_routing_skew(case, decode_weights):
    """Every token prefers the same few experts: segments of many rows beside empty
    ones (decode: 8 experts x 128 rows; prefill-like: 2 experts x T rows in the CTA-pair
    kernel), and with a capacity most routes are dropped."""
    if case == "decode_hot8":
        w = workloads.scaled(workloads.decode(128), logit_bias="hot8")
        layer, perm = run_and_check(w, weights=decode_weights, sample_rows=256, sample_tokens=32)
        assert sorted(np.nonzero(perm["counts"])[0].tolist()) == list(range(8))
    elif case == "tiny_hot2_capacity":
        w = workloads.scaled(workloads.tiny(), logit_bias="hot2")
        layer, perm = run_and_check(w)
        assert perm["counts"].tolist()[:2] == [80, 80] and perm["n_dropped"] == 2 * 256 - 160
    elif case == "prefill_hot2":
        w = workloads.scaled(workloads.prefill(), T=1024, d=512, I=1024, logit_bias="hot2")
        layer, perm = run_and_check(w, sample_rows=128, sample_tokens=48)
        assert perm["counts"].tolist() == [1024, 1024, 0, 0, 0, 0, 0, 0]
    else:
        w = workloads.scaled(workloads.v3(), T=384, d=256, I=128, shared_I=128,
                             logit_bias="hot8")
        layer, perm = run_and_check(w, sample_rows=128, sample_tokens=48)
        assert perm["n_dropped"] > 0


def test_tiny_full_gathered_rows():
    """The maps-only permute with the gathering gate/up loader gives the same checks."""
    run_and_check(workloads.tiny(), gather=True)


@pytest.mark.parametrize("T", [1, 32])
def test_decode_gathered_rows(T, decode_weights):
    run_and_check(workloads.decode(T), weights=decode_weights, sample_rows=4096, gather=True)


def test_v3_small_full_gathered_rows():
    w = workloads.scaled(workloads.v3(), T=64, d=256, I=256, shared_I=128)
    run_and_check(w, sample_rows=10**6, gather=True)


@pytest.mark.slow
def test_prefill_full_size_sampled():
    run_and_check(workloads.prefill(), sample_tokens=12, sample_rows=256, seed=2, every_tile=True)


@pytest.mark.slow
def test_v3_full_size_sampled():
    layer, perm = run_and_check(workloads.v3(), sample_tokens=6, sample_rows=256, seed=3,
                                every_tile=True)
    assert layer.capacity == 256
    # capacity 1.0 with a skewed selection bias must actually drop routes
    assert perm["n_dropped"] > 0


def test_v3_small_full():
    w = workloads.scaled(workloads.v3(), T=64, d=256, I=256, shared_I=128)
    run_and_check(w, sample_rows=10**6)


# ----------------------------------------------------------------------------
# FP8 dispatch payload ([M6.6] 0x0AB-0x0AC): E4M3 rows + fp32 scales permuted
# together, dequantized in the gate/up GEMM's loader
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("payload", ["fp8_row", "fp8_block128"])
def test_tiny_full_fp8(payload):
    run_and_check(workloads.tiny(), payload=payload)


@pytest.mark.parametrize("payload", ["fp8_row", "fp8_block128"])
def test_decode_T128_full_fp8(payload, decode_weights):
    run_and_check(workloads.decode(128), weights=decode_weights, sample_rows=4096, payload=payload)


@pytest.mark.parametrize("payload", ["fp8_row", "fp8_block128"])
def test_decode_T128_full_fp8_fused_loader(payload, decode_weights):
    """The gate/up pass dequantizing E4M3 tiles in its loader, in the layer."""
    layer, _ = run_and_check(workloads.decode(128), weights=decode_weights, sample_rows=4096,
                             payload=payload, fp8_loader="fused")
    assert layer.fused_fp8


@pytest.mark.parametrize("T", [1, 8])
def test_decode_fp8_fused_loader_small(T, decode_weights):
    run_and_check(workloads.decode(T), weights=decode_weights, sample_rows=4096,
                  payload="fp8_block128", fp8_loader="fused")


@pytest.mark.parametrize("payload", ["fp8_row", "fp8_block128"])
def test_v3_small_full_fp8(payload):
    w = workloads.scaled(workloads.v3(), T=64, d=384, I=256, shared_I=128)
    run_and_check(w, sample_rows=10**6, payload=payload)


@pytest.mark.slow
def test_v3_full_size_sampled_fp8():
    run_and_check(workloads.v3(), sample_tokens=6, sample_rows=256, seed=5, payload="fp8_block128")


@pytest.mark.slow
def test_prefill_full_size_sampled_fp8():
    run_and_check(workloads.prefill(), sample_tokens=8, sample_rows=256, seed=6, payload="fp8_row")


# ----------------------------------------------------------------------------
# pooled waves
# ----------------------------------------------------------------------------

def pooled_check(w, policy, sample_tokens, sample_rows, seed):
    import grouped_expert_gemm_gb300 as g
    logits, _ = workloads.make_router_inputs(w, DEV)
    x = workloads.make_activations(w, DEV)
    wg, wu, wd = workloads.make_expert_weights(w, DEV)
    pool_cap = g.capacity_from_factor(w.sender_cf, w.R, w.n_dest * w.n_waves)
    local_cap = g.capacity_from_factor(w.receiver_cf, w.R, w.local_per_dest * w.n_waves)
    assert pool_cap == oracle.pool_capacity(w.sender_cf, w.T, w.k, w.n_dest, w.n_waves)
    assert local_cap == oracle.local_capacity(w.receiver_cf, w.T, w.k, w.local_per_dest, w.n_waves)
    layer = g.PooledMoELayer(w.T, w.d, w.k, w.I, w.n_dest, w.local_per_dest, w.n_waves, pool_cap,
                             local_cap, wg, wu, wd, wave_policy=policy, device=DEV)
    pol = "stripe" if policy == g.MOE_WAVE_STRIPE else "destmod"
    layer.route(logits)
    torch.cuda.synchronize()
    ids, gates = oracle.route_softmax(host(logits), w.k)
    assert np.array_equal(host(layer.topk_ids), ids)
    assert_gates(host(layer.gates), gates)
    xb = bits(x)
    rng = np.random.default_rng(seed)
    tokens = np.sort(rng.choice(w.T, min(sample_tokens, w.T), replace=False))
    fetch = weights_fetcher(wg, wu, wd)
    ref_out = np.zeros((len(tokens), w.d))
    totals = dict(sender=0, receiver=0, accepted=0)
    for wave in range(w.n_waves):
        layer.pack(x, wave)
        layer.compact_wave(wave)
        layer.experts()
        layer.combine_wave(wave)
        torch.cuda.synchronize()
        assert int(layer.dev_status.item()) == 0
        rp = oracle.pool_pack(ids, xb, w.n_dest, w.local_per_dest, w.n_waves, pool_cap, wave, pol)
        hdr = bits(layer.pools[:, 0, :])
        assert np.array_equal(hdr, rp["pools"][:, 0, :])
        assert np.array_equal(host(layer.route_to_poolrow), rp["route_to_poolrow"])
        assert np.array_equal(host(layer.pool_fill), rp["fill"])
        assert int(host(layer.sender_drops)[wave]) == rp["sender_drops"]
        rc = oracle.pool_compact(rp["pools"], pool_cap, w.local_per_dest, local_cap)
        assert np.array_equal(host(layer.poolrow_to_row), rc["poolrow_to_row"])
        assert np.array_equal(host(layer.local_counts), rc["local_counts"])
        assert int(host(layer.receiver_drops)[wave]) == rc["receiver_drops"]
        comp = oracle.compose_map(rp["route_to_poolrow"], rc["poolrow_to_row"])
        assert np.array_equal(host(layer.route_to_row), comp)
        # payload rows: sampled bit copies in pools and in the compact arrays
        placed = np.nonzero(rp["route_to_poolrow"] >= 0)[0]
        if placed.size:
            pick = rng.choice(placed, min(sample_rows, placed.size), replace=False)
            pr = rp["route_to_poolrow"][pick]
            got_pool = bits(layer.pools.view(-1, w.d)[torch.from_numpy(
                (pr // pool_cap) * (pool_cap + 1) + 1 + pr % pool_cap).to(DEV)])
            assert np.array_equal(got_pool, xb[pick // w.k])
            cr = comp[pick]
            keep = cr >= 0
            got_c = bits(layer.compact[torch.from_numpy(cr[keep]).to(DEV)])
            assert np.array_equal(got_c, xb[pick[keep] // w.k])
        # H and y on rows reaching every 128-row m-tile of each local expert's array
        begins = np.arange(w.local_per_dest) * local_cap
        trows = stratified_rows(begins, rc["local_counts"], rng)
        assert_every_tile_reached(trows, begins, rc["local_counts"])
        route_of_row = np.full(w.local_per_dest * local_cap, -1)
        route_of_row[comp[comp >= 0]] = np.nonzero(comp >= 0)[0]
        assert np.all(route_of_row[trows] >= 0)
        h_ref, y_ref = oracle_expert_rows(trows, trows // local_cap,
                                          xb[route_of_row[trows] // w.k], fetch)
        idx = torch.from_numpy(trows).to(DEV)
        assert_float_parity(oracle.bf16_to_f64(bits(layer.H[idx])), h_ref,
                            f"pooled H on every m-tile, wave {wave}")
        assert_float_parity(oracle.bf16_to_f64(bits(layer.y[idx])), y_ref,
                            f"pooled y on every m-tile, wave {wave}")
        # sampled expert rows and this wave's contribution to the sampled tokens
        for i, t in enumerate(tokens):
            for j in range(w.k):
                row = comp[t * w.k + j]
                if row < 0:
                    continue
                l = row // local_cap
                wgl, wul, wdl = fetch(l)
                _, y = oracle.swiglu(oracle.bf16_to_f64(xb[t:t + 1]), oracle.bf16_to_f64(wgl),
                                     oracle.bf16_to_f64(wul), oracle.bf16_to_f64(wdl))
                got_y = oracle.bf16_to_f64(bits(layer.y[row:row + 1]))
                assert_float_parity(got_y, y, "pooled expert row")
                ref_out[i] += gates[t, j] * y[0]
        totals["sender"] += rp["sender_drops"]
        totals["receiver"] += rc["receiver_drops"]
        totals["accepted"] += int((comp >= 0).sum())
    assert totals["sender"] + totals["receiver"] + totals["accepted"] == w.R
    assert_float_parity(host(layer.out)[tokens], ref_out, "pooled combined output")
    return totals


@pytest.mark.parametrize("policy", [0, 1])
def test_pooled_small(policy):
    w = workloads.scaled(workloads.pooled(), T=2048, d=256, I=256, n_dest=32, E=32 * 6)
    pooled_check(w, policy, sample_tokens=64, sample_rows=512, seed=4)


@pytest.mark.slow
def test_pooled_full_size_sampled():
    totals = pooled_check(workloads.pooled(), 0, sample_tokens=8, sample_rows=256, seed=4)
    rates = oracle.drop_rates(65536 * 8, totals["sender"], totals["receiver"])
    assert 0 < rates["total"] < 0.5


# ----------------------------------------------------------------------------
# host-buffer pipeline: copies overlapped with the neighbouring steps' layer
# ----------------------------------------------------------------------------

def _host_steps(w, n, seed):
    out = []
    for i in range(n):
        wi = workloads.scaled(w, seed=seed + i)
        logits, _ = workloads.make_router_inputs(wi, DEV)
        x = workloads.make_activations(wi, DEV)
        out.append((logits.cpu().pin_memory(), x.cpu().pin_memory()))
    return out


@pytest.mark.parametrize("use_graph", [False, True])
def test_host_pipeline_equals_forward(use_graph):
    import grouped_expert_gemm_gb300 as g
    w = workloads.tiny()
    wg, wu, wd = workloads.make_expert_weights(w, DEV)
    layer = make_layer(w, wg, wu, wd)
    steps = _host_steps(w, 5, seed=40)
    outs = [torch.empty((w.T, w.d), dtype=torch.float32).pin_memory() for _ in steps]
    pipe = g.HostPipeline(layer)
    stream = torch.cuda.Stream(DEV)

    def run():
        pipe.begin(stream)
        for (lh, xh), oh in zip(steps, outs):
            pipe.submit(lh, xh, oh)
        pipe.end(stream)

    with torch.cuda.stream(stream):
        if use_graph:
            run()  # warm-up outside capture
            stream.synchronize()
            for o in outs:
                o.zero_()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                run()
            graph.replay()
        else:
            run()
    stream.synchronize()
    assert int(layer.dev_status.item()) == 0
    ref_layer = make_layer(w, wg, wu, wd)
    for (lh, xh), oh in zip(steps, outs):
        ref = ref_layer.forward(lh.to(DEV), xh.to(DEV))
        torch.cuda.synchronize()
        assert torch.equal(oh, ref.cpu())


def test_host_pipeline_pooled_layer():
    import grouped_expert_gemm_gb300 as g
    w = workloads.scaled(workloads.pooled(), T=1024, d=256, I=256, n_dest=32, E=32 * 6)
    wg, wu, wd = workloads.make_expert_weights(w, DEV)
    pool_cap = g.capacity_from_factor(w.sender_cf, w.R, w.n_dest * w.n_waves)
    local_cap = g.capacity_from_factor(w.receiver_cf, w.R, w.local_per_dest * w.n_waves)

    def mk():
        return g.PooledMoELayer(w.T, w.d, w.k, w.I, w.n_dest, w.local_per_dest, w.n_waves,
                                pool_cap, local_cap, wg, wu, wd, device=DEV)
    layer = mk()
    steps = _host_steps(w, 3, seed=50)
    outs = [torch.empty((w.T, w.d), dtype=torch.float32).pin_memory() for _ in steps]
    pipe = g.HostPipeline(layer)
    stream = torch.cuda.Stream(DEV)
    with torch.cuda.stream(stream):
        pipe.begin(stream)
        for (lh, xh), oh in zip(steps, outs):
            pipe.submit(lh, xh, oh)
        pipe.end(stream)
    stream.synchronize()
    ref_layer = mk()
    for (lh, xh), oh in zip(steps, outs):
        ref = ref_layer.forward(lh.to(DEV), xh.to(DEV))
        torch.cuda.synchronize()
        assert torch.equal(oh, ref.cpu())


def test_pooled_overlap_equals_the_sequential_schedule():
    """The overlapped pooled forward (pack, compact and combine on a second stream, wave
    buffers held twice) gives the sequential forward's output bit for bit, eagerly and
    replayed from a captured graph over changing inputs."""
    import grouped_expert_gemm_gb300 as g
    w = workloads.scaled(workloads.pooled(), T=2048, d=256, I=256, n_dest=32, E=32 * 6)
    wg, wu, wd = workloads.make_expert_weights(w, DEV)
    pool_cap = g.capacity_from_factor(w.sender_cf, w.R, w.n_dest * w.n_waves)
    local_cap = g.capacity_from_factor(w.receiver_cf, w.R, w.local_per_dest * w.n_waves)

    def mk(overlap):
        return g.PooledMoELayer(w.T, w.d, w.k, w.I, w.n_dest, w.local_per_dest, w.n_waves,
                                pool_cap, local_cap, wg, wu, wd, device=DEV, overlap=overlap)
    ov, seq = mk(True), mk(False)
    assert ov.overlap and not seq.overlap
    logits, _ = workloads.make_router_inputs(w, DEV)
    x = workloads.make_activations(w, DEV)
    ov.forward(logits, x)
    seq.forward(logits, x)
    torch.cuda.synchronize()
    assert int(ov.dev_status.item()) == 0
    assert torch.equal(ov.out, seq.out)
    assert torch.equal(ov.sender_drops, seq.sender_drops)
    assert torch.equal(ov.receiver_drops, seq.receiver_drops)
    # graph replays on new inputs
    stream = torch.cuda.Stream(DEV)
    lg = logits.clone()
    xx = x.clone()
    with torch.cuda.stream(stream):
        ov.forward(lg, xx)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        ov.forward(lg, xx)
    for seed in range(2):
        gen = torch.Generator(device=DEV).manual_seed(100 + seed)
        lg.copy_(torch.randn(lg.shape, generator=gen, device=DEV))
        xx.copy_(torch.randn(xx.shape, generator=gen, device=DEV).to(torch.bfloat16))
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            graph.replay()
        stream.synchronize()
        seq.forward(lg, xx)
        torch.cuda.synchronize()
        assert torch.equal(ov.out, seq.out)
