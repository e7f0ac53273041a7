"""Pins for the CPU oracle: values the pages print, closed forms, invariants and
brute force on tiny inputs.  None of these re-types the oracle's own formula;
each checks it against something independent of it.  CPU only.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import moe_oracle as om

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------------------
# Worked fixtures printed on the pages
# ----------------------------------------------------------------------------

def test_m62_loop9_count_prefix_permute():
    fx = load("m62_loop9_permute_combine.json")
    ids = np.array(fx["expert_of_route"]).reshape(-1, fx["k"])
    p = oracle.permute(ids, fx["E"], -1)
    assert p["counts"].tolist() == fx["counts"]
    assert p["offsets"].tolist() == fx["offsets"]
    assert p["row_to_route"].tolist() == fx["pi"]
    assert p["route_to_row"].tolist() == fx["inverse_pi"]
    assert p["n_dropped"] == 0


def test_m62_loop9_combine_with_scalar_experts():
    fx = load("m62_loop9_permute_combine.json")
    k, E = fx["k"], fx["E"]
    ids = np.array(fx["expert_of_route"]).reshape(-1, k)
    hidden = np.array(fx["hidden"], dtype=np.float64)
    p = oracle.permute(ids, E, -1)
    x_perm = hidden[p["row_to_route"] // k]
    scale = np.array(fx["scalar_expert"], dtype=np.float64)
    z = scale[ids.reshape(-1)[p["row_to_route"]]][:, None] * x_perm
    out = oracle.combine(z, p["route_to_row"], np.array(fx["gate_of_route"]), 4, k)
    np.testing.assert_allclose(out, np.array(fx["Y"]), rtol=0, atol=1e-12)


def test_m66_loop3_six_segments_and_combine():
    fx = load("m66_loop3_six_segments.json")
    k = fx["k"]
    slots = np.array(fx["physical_slot_of_route"]).reshape(-1, k)
    p = oracle.permute(slots, 6, -1)
    assert p["counts"].tolist() == fx["slot_counts"]
    assert p["offsets"].tolist() == fx["slot_offsets"]
    members = [p["row_to_route"][p["offsets"][q]:p["offsets"][q + 1]].tolist() for q in range(6)]
    assert members == fx["slot_members"]
    hidden = np.array(fx["hidden"], dtype=np.float64)
    logical = np.array(fx["logical_expert_of_slot"])
    scale = np.array(fx["scalar_expert"], dtype=np.float64)
    row_slot = slots.reshape(-1)[p["row_to_route"]]
    z = scale[logical[row_slot]][:, None] * hidden[p["row_to_route"] // k]
    out = oracle.combine(z, p["route_to_row"], np.array(fx["gate_of_route"]), 4, k)
    np.testing.assert_allclose(out, np.array(fx["Y"]), rtol=1e-12, atol=1e-12)


def test_m66_loop3_send_counts_and_offsets():
    """Count + exclusive prefix keyed by destination, per source rank."""
    fx = load("m66_loop3_six_segments.json")
    dst = np.array(fx["destination_rank_of_route"])
    src = np.array(fx["source_rank_of_route"])
    for p_rank in (0, 1):
        sel = dst[src == p_rank]
        perm = oracle.permute(sel.reshape(-1, 1), 4, -1)
        assert perm["counts"].tolist() == fx["send_counts"][p_rank]
        assert perm["offsets"].tolist() == fx["send_offsets"][p_rank]


def test_m66_runner_flop_ledger():
    fx = load("m66_loop3_six_segments.json")["runner_flops"]
    d, f = fx["d"], fx["d_ff"]
    assert oracle.swiglu_flops(fx["grouped_rows"], d, f) == fx["grouped"]
    assert oracle.swiglu_flops(fx["padded_rows"], d, f) == fx["padded"]
    assert oracle.swiglu_flops(fx["block_rows"], d, f) == fx["block"]


def _logit(p):
    return np.float32(np.log(np.asarray(p, np.float64) / (1.0 - np.asarray(p, np.float64))))


def test_m62_v3_group_gate_fixture():
    fx = load("m62_v3_group_gate.json")
    z = _logit(fx["affinity"])[None, :]
    ids, gates, groups, gscore = oracle.route_sigmoid_group(
        z, np.array(fx["bias"], np.float32), fx["k"], fx["n_group"], fx["topk_group"],
        fx["route_scale"], return_groups=True)
    assert ids[0].tolist() == fx["ids_with_bias"]
    assert groups[0].tolist() == fx["selected_groups_with_bias"]
    np.testing.assert_allclose(gscore[0], fx["group_top2_corrected"], atol=2e-6)
    np.testing.assert_allclose(gates[0], fx["gates_with_bias"], atol=1.5e-6)
    assert abs(gates[0].sum() - fx["route_scale"]) < 1e-12
    ids0, _, groups0, _ = oracle.route_sigmoid_group(
        z, None, fx["k"], fx["n_group"], fx["topk_group"], fx["route_scale"], return_groups=True)
    assert groups0[0].tolist() == fx["selected_groups_without_bias"]
    # without bias the four best affinities inside groups 2 and 1
    assert ids0[0].tolist() == [6, 7, 3, 4]


def test_m62_v3_fixture_detects_planted_tie_break(monkeypatch):
    """Plant a wrong tie-break in the oracle: the page's 0.65 tie must catch it."""
    fx = load("m62_v3_group_gate.json")
    z = _logit(fx["affinity"])[None, :]

    def highest_index_first(scores):
        rev = scores[..., ::-1]
        o = np.argsort(-rev, axis=-1, kind="stable")
        return scores.shape[-1] - 1 - o
    monkeypatch.setattr(om, "_order_desc_lowest_index", highest_index_first)
    ids, _ = om.route_sigmoid_group(z, np.array(fx["bias"], np.float32), fx["k"],
                                    fx["n_group"], fx["topk_group"], fx["route_scale"])
    assert ids[0].tolist() != fx["ids_with_bias"]


def test_m62_v3_fixture_detects_planted_gate_source(monkeypatch):
    """Plant 'gates from corrected scores': expert 1's gate turns into the page's 0.552721."""
    fx = load("m62_v3_group_gate.json")
    z = _logit(fx["affinity"])[None, :]
    bias = np.array(fx["bias"], np.float32)
    real = om.sigmoid_det_f32
    calls = {"n": 0}

    def corrected_sigmoid(v):
        return (real(v) + bias).astype(np.float32)
    monkeypatch.setattr(om, "sigmoid_det_f32", corrected_sigmoid)
    # selection with zero extra bias now sees s~ and the gate uses s~ as well
    ids, gates = om.route_sigmoid_group(z, np.zeros(12, np.float32), fx["k"], fx["n_group"],
                                        fx["topk_group"], fx["route_scale"])
    assert ids[0].tolist() == fx["ids_with_bias"]
    assert abs(gates[0][3] - fx["gate_of_expert1_if_corrected_scores_reused"]) < 1.5e-6
    assert abs(gates[0][3] - fx["gates_with_bias"][3]) > 0.4


def test_pool_capacities_shapes_and_sizes():
    fx = load("pool_capacity_and_sizes.json")
    T, k = fx["tokens"], fx["top_k"]
    assert T * k == fx["assignments"]
    assert oracle.pool_capacity(fx["sender_cf"], T, k, fx["n_dest"], fx["n_waves"]) == fx["pool_cap"]
    assert oracle.local_capacity(fx["receiver_cf"], T, k, fx["local_per_dest"],
                                 fx["n_waves"]) == fx["local_cap"]
    gib = lambda shape: float(np.prod(shape)) * 2 / 2**30
    assert round(gib(fx["sender_pool_shape"]), 2) == fx["sender_pool_gib"]
    assert round(gib(fx["receiver_compact_shape"]), 2) == fx["receiver_compact_gib"]
    assert round(gib(fx["historical_direct_shape"]), 2) == fx["historical_direct_gib"]
    D, L = oracle.expert_to_dest_local(np.array(fx["owner_example"]["experts"]), fx["local_per_dest"])
    assert set(D.tolist()) == {fx["owner_example"]["gpu"]}
    assert L.tolist() == list(range(6))
    # the pools carry one extra header row: the all-to-all shape
    ids = np.zeros((4, 1), dtype=np.int64)
    x = np.zeros((4, fx["width"]), dtype=np.uint16)
    pk = oracle.pool_pack(ids, x, fx["n_dest"], fx["local_per_dest"], fx["n_waves"],
                          fx["pool_cap"], 0)
    assert list(pk["pools"].shape) == fx["a2a_shape_with_header"]


def test_drop_rate_definitions():
    fx = load("pool_capacity_and_sizes.json")["drop_example"]
    total = 10**6
    r = oracle.drop_rates(total, round(fx["sender_pct"] * total / 100), round(fx["receiver_pct"] * total / 100))
    assert abs(r["total"] * 100 - fx["total_pct"]) < 1e-9
    # the page's 13.12% was evidently taken from unrounded rates; rounded inputs give 13.13%
    assert abs(r["receiver_conditional"] * 100 - fx["conditional_receiver_pct"]) < 0.015


def test_capacity_values_of_the_workloads():
    assert oracle.capacity(1.25, 256, 2, 8) == 80
    assert oracle.capacity(1.0, 8192, 8, 256) == 256
    assert oracle.capacity(1.0, 7, 1, 7) == 1
    assert oracle.capacity(1.1, 10, 1, 1) == 11  # 11.000... on paper, not 12


def test_staging_bytes_ledger():
    """[M6.2] 0x03E: N=4096, k=2, d=4096, bf16 -> 64 MiB of all-route activation rows."""
    T, k, d = 4096, 2, 4096
    assert T * k * d * 2 == 64 * 2**20


# ----------------------------------------------------------------------------
# Routing: brute force and closed forms
# ----------------------------------------------------------------------------

def _py_topk(row, k):
    """Selection sort with the explicit key (value desc, index asc)."""
    chosen = []
    for _ in range(k):
        best = None
        for e, v in enumerate(row):
            if e in chosen:
                continue
            if best is None or v > row[best] or (v == row[best] and e < best):
                best = e
        chosen.append(best)
    return chosen


def test_route_softmax_brute_force_with_ties():
    rng = np.random.default_rng(0)
    values = np.array([-1.0, -0.0, 0.0, 0.5, 0.5, 2.0], dtype=np.float32)
    for _ in range(300):
        T, E = rng.integers(1, 5), rng.integers(1, 7)
        k = int(rng.integers(1, E + 1))
        z = rng.choice(values, size=(T, E)).astype(np.float32)
        ids, gates = oracle.route_softmax(z, k)
        for t in range(T):
            exp_ids = _py_topk(z[t].tolist(), k)
            assert ids[t].tolist() == exp_ids
            ev = [math.exp(float(z[t, e]) - float(z[t, exp_ids[0]])) for e in exp_ids]
            s = sum(ev)
            assert np.allclose(gates[t], [v / s for v in ev], rtol=1e-14, atol=0)


def test_route_softmax_k_equals_E_is_full_softmax():
    from scipy.special import softmax
    rng = np.random.default_rng(1)
    z = rng.standard_normal((64, 8)).astype(np.float32)
    ids, gates = oracle.route_softmax(z, 8)
    full = softmax(z.astype(np.float64), axis=1)
    np.testing.assert_allclose(gates, np.take_along_axis(full, ids, 1), rtol=1e-13)
    assert np.all(np.diff(np.take_along_axis(z, ids, 1), axis=1) <= 0)


def test_route_softmax_gates_sum_to_one():
    rng = np.random.default_rng(2)
    z = rng.standard_normal((128, 128)).astype(np.float32)
    _, gates = oracle.route_softmax(z, 8)
    np.testing.assert_allclose(gates.sum(1), 1.0, rtol=1e-14)


def _py_route_group(s_row, st_row, n_group, topk_group, k, scale):
    E = len(st_row)
    gs = E // n_group
    gscores = []
    for g in range(n_group):
        members = list(range(g * gs, (g + 1) * gs))
        vals = [st_row[e] for e in members]
        top = _py_topk(vals, 2)
        gscores.append(np.float32(np.float32(vals[top[0]]) + np.float32(vals[top[1]])))
    keep = _py_topk(gscores, topk_group)
    masked = [st_row[e] if (e // gs) in keep else -math.inf for e in range(E)]
    ids = _py_topk(masked, k)
    ssum = sum(float(s_row[e]) for e in ids)
    return ids, [scale * float(s_row[e]) / ssum for e in ids]


def test_route_sigmoid_group_brute_force():
    rng = np.random.default_rng(3)
    for _ in range(200):
        n_group = int(rng.integers(2, 5))
        gs = int(rng.integers(2, 4))
        E = n_group * gs
        topk_group = int(rng.integers(1, n_group + 1))
        k = int(rng.integers(1, topk_group * gs + 1))
        T = 3
        z = rng.choice(np.array([-1.0, 0.0, 0.3, 0.3, 1.5], np.float32), size=(T, E))
        b = rng.choice(np.array([0.0, 0.1, -0.1], np.float32), size=E)
        ids, gates = oracle.route_sigmoid_group(z, b, k, n_group, topk_group, 2.5)
        s = oracle.sigmoid_det_f32(z)
        st = (s + b).astype(np.float32)
        for t in range(T):
            e_ids, e_g = _py_route_group(s[t].tolist(), st[t].tolist(), n_group, topk_group, k, 2.5)
            assert ids[t].tolist() == e_ids
            np.testing.assert_allclose(gates[t], e_g, rtol=1e-13)


def test_sigmoid_det_accuracy_and_shape():
    rng = np.random.default_rng(4)
    z = np.concatenate([rng.standard_normal(200000) * 4, rng.uniform(-90, 90, 200000),
                        [0.0, -0.0, 1e-30, -1e-30, 87.0, -87.0, 100.0, -100.0]]).astype(np.float32)
    s = oracle.sigmoid_det_f32(z)
    exact = 1.0 / (1.0 + np.exp(-z.astype(np.float64)))
    inside = np.abs(z) <= 87
    ulp = np.spacing(exact[inside].astype(np.float32)).astype(np.float64)
    err = np.abs(s[inside] - exact[inside]) / ulp
    assert err.max() <= 4.0, err.max()
    assert oracle.sigmoid_det_f32(np.float32(0.0)) == np.float32(0.5)
    zs = np.sort(z)
    assert np.all(np.diff(oracle.sigmoid_det_f32(zs).astype(np.float64)) >= 0)
    assert np.all((s >= 0) & (s <= 1))


def test_exp_det_matches_exp_to_a_few_ulp():
    x = np.linspace(-87, 87, 400001).astype(np.float32)
    got = oracle.exp_det_f32(x).astype(np.float64)
    ref = np.exp(x.astype(np.float64))
    ulp = np.spacing(ref.astype(np.float32)).astype(np.float64)
    assert (np.abs(got - ref) / ulp).max() <= 3.0


# ----------------------------------------------------------------------------
# Permute: brute force and invariants
# ----------------------------------------------------------------------------

def _py_permute(ids, E, cap):
    flat = [int(v) for v in np.asarray(ids).reshape(-1)]
    seen = [0] * E
    accepted = []
    for r, e in enumerate(flat):
        if cap < 0 or seen[e] < cap:
            accepted.append(r)
        seen[e] += 1
    rows = sorted(accepted, key=lambda r: (flat[r], r))
    counts = [sum(1 for r in accepted if flat[r] == e) for e in range(E)]
    r2r = [-1] * len(flat)
    for row, r in enumerate(rows):
        r2r[r] = row
    return rows, r2r, counts


@pytest.mark.parametrize("cap", [-1, 0, 1, 2, 3, 100])
def test_permute_brute_force(cap):
    rng = np.random.default_rng(5 + cap)
    for _ in range(100):
        T, E = int(rng.integers(0, 6)), int(rng.integers(1, 7))
        k = int(rng.integers(1, min(E, 3) + 1))
        ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]) if T else np.zeros((0, k), int)
        p = oracle.permute(ids, E, cap)
        rows, r2r, counts = _py_permute(ids, E, cap)
        assert p["row_to_route"].tolist() == rows
        assert p["route_to_row"].tolist() == r2r
        assert p["counts"].tolist() == counts
        assert p["offsets"].tolist() == [0] + list(np.cumsum(counts))
        assert p["n_dropped"] + sum(counts) == T * k
        acc = p["route_to_row"] >= 0
        assert np.all(p["row_to_route"][p["route_to_row"][acc]] == np.nonzero(acc)[0])
        if cap >= 0:
            assert all(c <= cap for c in counts)


def test_permute_rejects_bad_ids():
    with pytest.raises(ValueError):
        oracle.permute(np.array([[0, 5]]), 4, -1)


# ----------------------------------------------------------------------------
# SwiGLU and combine: special cases with independent answers
# ----------------------------------------------------------------------------

def test_f64_to_bf16_matches_torch_on_fp32_values():
    rng = np.random.default_rng(6)
    v = np.concatenate([rng.standard_normal(100000).astype(np.float32),
                        (rng.standard_normal(1000) * 1e-39).astype(np.float32),
                        np.array([1.00390625, 1.01171875, -2.0, 0.0, -0.0, 3.0e38], np.float32)])
    ours = oracle.f64_to_bf16(v.astype(np.float64))
    theirs = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, theirs)
    assert np.array_equal(oracle.f64_to_bf16(oracle.bf16_to_f64(ours)), ours)


def test_swiglu_closed_form_scalar():
    x, wg, wu, wd = 2.0, 0.5, 3.0, 0.25
    h, y = oracle.swiglu(np.array([[x]]), np.array([[wg]]), np.array([[wu]]), np.array([[wd]]),
                         round_h=False, round_y=False)
    g, u = x * wg, x * wu
    expect_h = g / (1 + math.exp(-g)) * u
    assert abs(h[0, 0] - expect_h) < 1e-14
    assert abs(y[0, 0] - expect_h * wd) < 1e-14


def test_grouped_rows_use_each_segments_own_expert():
    """Several segments with distinct scalar experts (d = I = 1): every row's h and y
    equal the closed form of its own segment's expert, each rounded to bf16 by torch,
    so a segment/expert mix-up, a shifted segment start or a dropped row fails."""
    # expert q: (wg, wu, wd); values exact in bf16 and distinct per expert
    experts = [(0.5, 3.0, 0.25), (-1.0, 2.0, 0.5), (2.0, -0.5, -1.5), (0.75, 1.25, 4.0)]
    begins, counts = [0, 3, 3, 7], [3, 0, 4, 2]    # segment 1 is empty, 2 starts at row 3
    xs = [1.0, -2.0, 0.5, 3.0, -0.25, 1.5, 2.5, -1.0, 0.125]
    to_bits = lambda v: torch.tensor(v, dtype=torch.float64).to(torch.bfloat16).view(
        torch.int16).numpy().view(np.uint16)
    x = to_bits([[v] for v in xs])
    wg = to_bits([[[e[0]]] for e in experts])
    wu = to_bits([[[e[1]]] for e in experts])
    wd = to_bits([[[e[2]]] for e in experts])
    y, h = oracle.grouped_swiglu_rows(x, begins, counts, wg, wu, wd)
    rows = [r for b, c in zip(begins, counts) for r in range(b, b + c)]
    assert sorted(y) == rows and sorted(h) == rows
    for q, (b, c) in enumerate(zip(begins, counts)):
        g_w, u_w, d_w = experts[q]
        for r in range(b, b + c):
            g, u = xs[r] * g_w, xs[r] * u_w
            h_ref = to_bits(g / (1.0 + math.exp(-g)) * u)
            y_ref = to_bits(float(torch.from_numpy(h_ref.view(np.int16)).view(torch.bfloat16)
                                  .to(torch.float64)) * d_w)
            assert h[r].tolist() == [int(h_ref)], (q, r)
            assert y[r].tolist() == [int(y_ref)], (q, r)


def test_dense_reduction_matches_independent_library():
    """E = k = 1 dropless: the layer is one dense SwiGLU FFN (checked with torch CPU fp64)."""
    rng = np.random.default_rng(7)
    T, d, I = 16, 64, 96
    x = oracle.f64_to_bf16(rng.standard_normal((T, d)))
    wg = oracle.f64_to_bf16(rng.standard_normal((1, d, I)) / 8)
    wu = oracle.f64_to_bf16(rng.standard_normal((1, d, I)) / 8)
    wd = oracle.f64_to_bf16(rng.standard_normal((1, I, d)) / 10)
    ids = np.zeros((T, 1), np.int64)
    p = oracle.permute(ids, 1, -1)
    xp = oracle.gather_rows(x, p["row_to_route"], 1)
    y, _ = oracle.grouped_swiglu_rows(xp, [0], [T], wg, wu, wd)
    ybits = np.stack([y[r] for r in range(T)])
    ids_g, gates = oracle.route_softmax(np.zeros((T, 1), np.float32), 1)
    out = oracle.combine(oracle.bf16_to_f64(ybits), p["route_to_row"], gates, T, 1)
    tx = torch.from_numpy(oracle.bf16_to_f64(x))
    tg = torch.from_numpy(oracle.bf16_to_f64(wg[0]))
    tu = torch.from_numpy(oracle.bf16_to_f64(wu[0]))
    td = torch.from_numpy(oracle.bf16_to_f64(wd[0]))
    h = torch.nn.functional.silu(tx @ tg) * (tx @ tu)
    h = h.to(torch.float32).to(torch.bfloat16).to(torch.float64)
    ref = (h @ td).numpy()
    # independent path rounds via fp32 (double rounding): allow one bf16 ulp of difference
    assert np.max(np.abs(out - ref) / (np.abs(ref) + 1e-3)) < 1e-2
    assert np.linalg.norm(out - ref) / np.linalg.norm(ref) < 2e-3


def test_fused_shared_experts_equal_their_sum():
    """[M6.2] 0x04C1: two shared experts fused into one wider SwiGLU equal their sum."""
    rng = np.random.default_rng(8)
    n, d, I = 5, 32, 48
    x = rng.standard_normal((n, d))
    ws = [(rng.standard_normal((d, I)), rng.standard_normal((d, I)), rng.standard_normal((I, d)))
          for _ in range(2)]
    ys = [oracle.swiglu(x, *w, round_h=False, round_y=False)[1] for w in ws]
    fused = oracle.swiglu(x, np.concatenate([ws[0][0], ws[1][0]], 1),
                          np.concatenate([ws[0][1], ws[1][1]], 1),
                          np.concatenate([ws[0][2], ws[1][2]], 0), round_h=False, round_y=False)[1]
    np.testing.assert_allclose(fused, ys[0] + ys[1], rtol=1e-12, atol=1e-10)


def test_combine_drops_accumulate_and_shared():
    rng = np.random.default_rng(9)
    T, k, d = 6, 3, 4
    y = rng.standard_normal((10, d))
    r2r = np.array([0, -1, 2, 3, 4, 5, -1, -1, -1, 6, 7, 8, 9, -1, 1, 2, 3, 4])
    g = rng.uniform(0, 1, T * k)
    sh = rng.standard_normal((T, d))
    init = rng.standard_normal((T, d))
    out = oracle.combine(y, r2r, g, T, k, shared_y_f64=sh, out_init=init)
    for t in range(T):
        ref = init[t] + sh[t]
        for j in range(k):
            r = r2r[t * k + j]
            if r >= 0:
                ref = ref + g[t * k + j] * y[r]
        np.testing.assert_allclose(out[t], ref, rtol=1e-13)
    assert np.allclose(out[2] - init[2] - sh[2], 0)  # a fully dropped token gets nothing routed


# ----------------------------------------------------------------------------
# Pooled layout: brute force and conservation
# ----------------------------------------------------------------------------

def _py_pack(ids, n_dest, L, n_waves, cap, wave, policy):
    flat = [int(v) for v in np.asarray(ids).reshape(-1)]
    seen = [0] * n_dest
    fill = [0] * n_dest
    hdr = [[0xFFFF] * cap for _ in range(n_dest)]
    where, drops = [-1] * len(flat), 0
    for r, e in enumerate(flat):
        D, l = e // L, e % L
        j = seen[D]
        seen[D] += 1
        w, row = (j % n_waves, j // n_waves) if policy == "stripe" else (D % n_waves, j)
        if w != wave:
            continue
        if row < cap:
            hdr[D][row] = l
            where[r] = D * cap + row
            fill[D] += 1
        else:
            drops += 1
    return hdr, where, fill, drops


def _py_compact(hdr, cap, n_local, local_cap):
    cnt = [0] * n_local
    out = [-1] * (len(hdr) * cap)
    drops = 0
    for s in range(len(hdr)):
        for r in range(cap):
            l = hdr[s][r]
            if l >= n_local:
                continue
            if cnt[l] < local_cap:
                out[s * cap + r] = l * local_cap + cnt[l]
            else:
                drops += 1
            cnt[l] += 1
    return out, [min(c, local_cap) for c in cnt], drops


@pytest.mark.parametrize("policy", ["stripe", "destmod"])
def test_pool_pack_compact_brute_force(policy):
    rng = np.random.default_rng(10)
    for _ in range(60):
        n_dest, L, n_waves = int(rng.integers(1, 5)), int(rng.integers(1, 4)), int(rng.integers(1, 4))
        E = n_dest * L
        T = int(rng.integers(1, 12))
        k = int(rng.integers(1, min(E, 3) + 1))
        ids = np.stack([rng.permutation(E)[:k] for _ in range(T)])
        d = 4
        x = rng.integers(0, 2**15, size=(T, d)).astype(np.uint16)
        cap = int(rng.integers(1, 5))
        lcap = int(rng.integers(1, 6))
        total_s = total_r = total_acc = 0
        for wave in range(n_waves):
            pk = oracle.pool_pack(ids, x, n_dest, L, n_waves, cap, wave, policy)
            hdr, where, fill, drops = _py_pack(ids, n_dest, L, n_waves, cap, wave, policy)
            assert pk["pools"][:, 0, :cap].tolist() == hdr
            assert pk["route_to_poolrow"].tolist() == where
            assert pk["fill"].tolist() == fill
            assert pk["sender_drops"] == drops
            for r, pr in enumerate(where):
                if pr >= 0:
                    assert pk["pools"][pr // cap, 1 + pr % cap].tolist() == x[r // k].tolist()
            cp = oracle.pool_compact(pk["pools"], cap, L, lcap)
            p2r, counts, rdrops = _py_compact(hdr, cap, L, lcap)
            assert cp["poolrow_to_row"].tolist() == p2r
            assert cp["local_counts"].tolist() == counts
            assert cp["receiver_drops"] == rdrops
            for i, row in enumerate(p2r):
                if row >= 0:
                    s, rr = divmod(i, cap)
                    assert np.array_equal(cp["compact"][row // lcap, row % lcap], pk["pools"][s, 1 + rr])
            composed = oracle.compose_map(pk["route_to_poolrow"], cp["poolrow_to_row"])
            total_s += drops
            total_r += rdrops
            total_acc += int((composed >= 0).sum())
        assert total_s + total_r + total_acc == T * k


def _py_compact_rotated(hdr, cap, n_local, local_cap, first):
    """Brute force of the rotated visit: sources first, first+1, ..., wrapping."""
    n_src = len(hdr)
    cnt = [0] * n_local
    out = [-1] * (n_src * cap)
    drops = 0
    for j in range(n_src):
        s_ = (first + j) % n_src
        for r in range(cap):
            l = hdr[s_][r]
            if l >= n_local:
                continue
            if cnt[l] < local_cap:
                out[s_ * cap + r] = l * local_cap + cnt[l]
            else:
                drops += 1
            cnt[l] += 1
    return out, [min(c, local_cap) for c in cnt], drops


def test_pool_compact_rotation_brute_force():
    """[POOL] 07's proposed per-receiver rotation: the overflow falls on the sources
    visited last, whichever they are."""
    rng = np.random.default_rng(12)
    for _ in range(40):
        n_src, cap, n_local = int(rng.integers(1, 6)), int(rng.integers(1, 5)), int(rng.integers(1, 4))
        lcap = int(rng.integers(1, 5))
        pools = np.zeros((n_src, cap + 1, 4), np.uint16)
        pools[:, 0, :] = 0xFFFF
        for s_ in range(n_src):
            fill = int(rng.integers(0, cap + 1))
            pools[s_, 0, :fill] = rng.integers(0, n_local, fill)
        hdr = pools[:, 0, :cap].tolist()
        for first in range(n_src):
            cp = oracle.pool_compact(pools, cap, n_local, lcap, first)
            p2r, counts, drops = _py_compact_rotated(hdr, cap, n_local, lcap, first)
            assert cp["poolrow_to_row"].tolist() == p2r
            assert cp["local_counts"].tolist() == counts
            assert cp["receiver_drops"] == drops
        # no rotation is the fixed source order
        base = oracle.pool_compact(pools, cap, n_local, lcap)
        assert base["poolrow_to_row"].tolist() == _py_compact(hdr, cap, n_local, lcap)[0]
    with pytest.raises(ValueError):
        oracle.pool_compact(np.zeros((2, 3, 4), np.uint16), 2, 1, 1, 2)


def test_pool_compact_skips_invalid_header_ids():
    pools = np.zeros((2, 4, 3), np.uint16)
    pools[:, 0, :] = 0xFFFF
    pools[0, 0, :3] = [0, 7, 1]
    pools[1, 0, :2] = [1, 1]
    cp = oracle.pool_compact(pools, 3, 2, 8)
    assert cp["bad_headers"] == 1
    assert cp["poolrow_to_row"].tolist() == [0, -1, 8, 9, 10, -1]
    assert cp["local_counts"].tolist() == [1, 3]


def test_compose_map_brute_force():
    rng = np.random.default_rng(11)
    a = rng.integers(-1, 10, 50)
    b = rng.integers(-1, 100, 10)
    out = oracle.compose_map(a, b)
    for i in range(50):
        assert out[i] == (-1 if a[i] < 0 else b[a[i]])


# ----------------------------------------------------------------------------
# Backward of the transpose, load telemetry and the bias controller
# ----------------------------------------------------------------------------

def test_m62_loop9_backward_of_the_transpose():
    """[M6.2] 0x03D: all-ones upstream gradient on the Loop 9 fixture."""
    fx = load("m62_loop9_permute_combine.json")
    k, E = fx["k"], fx["E"]
    ids = np.array(fx["expert_of_route"]).reshape(-1, k)
    hidden = np.array(fx["hidden"], dtype=np.float64)
    gates = np.array(fx["gate_of_route"])
    p = oracle.permute(ids, E, -1)
    x_perm = hidden[p["row_to_route"] // k]
    scale = np.array(fx["scalar_expert"], dtype=np.float64)
    row_expert = ids.reshape(-1)[p["row_to_route"]]
    z = scale[row_expert][:, None] * x_perm
    dy, dg = oracle.combine_backward(np.ones((4, 3)), z, p["route_to_row"], gates, 4, k)
    assert np.allclose(dg.reshape(-1), fx["backward_all_ones"]["gate_grad_by_route"], atol=1e-12)
    # scalar experts: dL/ds_e = sum over its rows of <dy_row, x_row>
    ds = [float(np.sum(dy[row_expert == e] * x_perm[row_expert == e])) for e in range(E)]
    np.testing.assert_allclose(ds, [15, 17.25, 10.2, 35.55], atol=1e-12)
    # route-input gradients s_e * dy, summed back to tokens through the inverse
    dx = oracle.unpermute_grad(scale[row_expert][:, None] * dy, p["route_to_row"], 4, k)
    np.testing.assert_allclose(dx, np.array([2.4, 2.4, 2.35, 3.5])[:, None] * np.ones((4, 3)),
                               atol=1e-12)


def test_combine_backward_is_the_adjoint_of_combine():
    """<combine(y), dout> = <y, dy> + sum_g dgates * gates-derivative (linearity checks)."""
    rng = np.random.default_rng(12)
    T, k, d, rows = 7, 3, 5, 25
    y = rng.standard_normal((rows, d))
    r2r = rng.permutation(rows)[: T * k]
    r2r[[2, 9]] = -1
    g = rng.uniform(0, 1, T * k)
    dout = rng.standard_normal((T, d))
    dy, dg = oracle.combine_backward(dout, y, r2r, g, T, k)
    out = oracle.combine(y, r2r, g, T, k)
    # out is linear in y: <out, dout> == <y, dy>
    assert abs(np.sum(out * dout) - np.sum(y * dy)) < 1e-10
    # and linear in the gates: <out, dout> == <g, dgates>
    assert abs(np.sum(out * dout) - np.sum(g.reshape(T, k) * dg)) < 1e-10
    # finite difference in one gate
    eps = 1e-6
    g2 = g.copy()
    g2[4] += eps
    fd = (np.sum(oracle.combine(y, r2r, g2, T, k) * dout) - np.sum(out * dout)) / eps
    assert abs(fd - dg.reshape(-1)[4]) < 1e-5


def test_unpermute_grad_is_the_adjoint_of_the_gather():
    rng = np.random.default_rng(13)
    T, k, d, E = 9, 2, 4, 5
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    p = oracle.permute(ids, E, 2)
    x = rng.standard_normal((T, d))
    xp = x[p["row_to_route"] // k]
    dxp = rng.standard_normal(xp.shape)
    dx = oracle.unpermute_grad(dxp, p["route_to_row"], T, k)
    assert abs(np.sum(xp * dxp) - np.sum(x * dx)) < 1e-10


def test_m62_skew_summaries_fixture():
    fx = load("m62_load_and_controller.json")
    for axis, (counts, cv2) in fx["cv2_by_axis"].items():
        assert abs(oracle.load_stats(counts)["cv2"] - cv2) < 1e-12, axis
    mv = fx["maxvio_toy"]
    assert abs(oracle.load_stats(mv["counts"])["max_vio"] - mv["max_vio"]) < 1e-12
    # closed forms: uniform counts and a single occupied unit
    u = oracle.load_stats([5] * 8)
    assert abs(u["h_norm"] - 1) < 1e-12 and abs(u["e_eff"] - 8) < 1e-9 and u["cv2"] == 0
    one = oracle.load_stats([0, 0, 7, 0])
    assert one["h_norm"] == 0 and abs(one["e_eff"] - 1) < 1e-12 and one["rho_max"] == 4
    assert oracle.load_stats([0, 0, 0])["total"] == 0


def test_m62_controller_step_fixture():
    fx = load("m62_load_and_controller.json")["controller"]
    c = np.array(fx["counts"])
    assert abs(c.mean() - fx["mean"]) < 1e-15
    b0 = np.zeros(c.size, np.float32)
    b1 = oracle.bias_update(b0, c, fx["gamma"], "sign")
    for e in fx["decrease"]:
        assert b1[e] == np.float32(-0.001)
    for e in fx["increase_zero_load"]:
        assert b1[e] == np.float32(0.001)
    assert np.all(np.sign(b1) == np.sign(c.mean() - c))
    bp = oracle.bias_update(b0, c, 0.01, "proportional")
    np.testing.assert_allclose(bp, 0.01 * (c.mean() - c), rtol=1e-6)


# ----------------------------------------------------------------------------
# FP8 dispatch payload ([M6.6] 0x0AB-0x0AF)
# ----------------------------------------------------------------------------

def test_m66_payload_ledger_table():
    fx = load("m66_fp8_payload_ledger.json")
    for row in fx["table"]:
        for mode in ("bf16", "fp8_row", "fp8_block"):
            assert oracle.payload_bytes(fx["rows"], row["d"], mode, fx["group"]) == row[mode], (row, mode)
    # the d = 3 row: fp8 plus scales is larger than bf16
    assert oracle.payload_bytes(6, 3, "fp8_row") > oracle.payload_bytes(6, 3, "bf16")


def _torch_e4m3_decode(codes):
    return torch.from_numpy(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e4m3_decode_matches_library_format_on_every_code():
    codes = np.arange(256, dtype=np.uint8)
    mine = om.e4m3_decode(codes)
    lib = _torch_e4m3_decode(codes)
    assert np.array_equal(np.isnan(mine), np.isnan(lib))
    fin = ~np.isnan(lib)
    assert np.array_equal(mine[fin], lib[fin])
    assert np.array_equal(np.signbit(mine[fin]), np.signbit(lib[fin]))
    # format landmarks: 2 NaN codes, 254 finite, largest 448, smallest normal 2^-6, subnormal 2^-9
    assert np.isnan(mine).sum() == 2 and np.nanmax(mine) == 448.0
    assert mine[0x08] == 2.0 ** -6 and mine[0x01] == 2.0 ** -9 and mine[0x38] == 1.0


def test_e4m3_encode_matches_library_rounding_in_range():
    """Nearest-even rounding against the library conversion on every code value,
    every midpoint (the ties), one fp32 ulp either side of each midpoint and random
    values; the library does not saturate, so only |v| < 464 is compared there."""
    pos = om.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = (pos[:-1] + pos[1:]) / 2
    mids32 = mids.astype(np.float32)
    assert np.array_equal(mids32.astype(np.float64), mids)  # midpoints are fp32-exact
    up = np.nextafter(mids32, np.float32(np.inf))
    dn = np.nextafter(mids32, np.float32(0))
    rng = np.random.default_rng(0)
    rnd = np.concatenate([rng.uniform(0, 463, 20000), rng.uniform(0, 2 ** -5, 5000)]).astype(np.float32)
    v = np.concatenate([pos, mids32, up, dn, rnd, [463.99]]).astype(np.float32)
    v = np.concatenate([v, -v])
    mine = om.e4m3_encode(v)
    lib = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(mine, lib)


def test_e4m3_encode_saturates_and_keeps_nan():
    v = np.array([448.0, 464.0, 465.0, 1e6, 3e38, -1e9, np.nan], np.float32)
    assert om.e4m3_encode(v).tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x7F]


def _bf16_rows(rng, n, d, scale=1.0):
    return oracle.f64_to_bf16(rng.standard_normal((n, d)) * scale)


@pytest.mark.parametrize("group,d", [(0, 64), (128, 256), (128, 200), (0, 3), (128, 3)])
def test_quantize_invariants(group, d):
    rng = np.random.default_rng(d + group)
    xb = _bf16_rows(rng, 9, d)
    xb[3] = 0  # an all-zero row
    xb[4, : min(d, 100)] = oracle.f64_to_bf16(rng.standard_normal(min(d, 100)) * 1e-3)
    q, s = oracle.quantize_fp8(xb, group)
    G = oracle.n_scale_groups(d, group)
    assert s.shape == (9, G) and q.shape == (9, d)
    g = d if group == 0 else group
    x = oracle.bf16_to_f64(xb)
    dec = om.e4m3_decode(q)
    for i in range(9):
        for j in range(G):
            blk = x[i, j * g:(j + 1) * g]
            amax = np.abs(blk).max()
            if amax == 0:
                assert s[i, j] == 1.0 and np.all(q[i, j * g:(j + 1) * g] & 0x7F == 0)
                continue
            # the scale maps the group's largest magnitude onto the largest code
            assert abs(float(s[i, j]) * 448 - amax) <= amax * 2 ** -23
            big = np.argmax(np.abs(blk))
            assert q[i, j * g + big] & 0x7F == 0x7E
            # every code is the nearest E4M3 value to x / s (brute force over all codes)
            ratio = blk / float(s[i, j])
            allv = om.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
            dist = np.abs(np.abs(ratio)[:, None] - allv[None, :]).min(axis=1)
            got = np.abs(np.abs(ratio) - np.abs(dec[i, j * g:(j + 1) * g]))
            assert np.all(got <= dist + 1e-6 * np.abs(ratio))
            assert np.all(np.sign(dec[i, j * g:(j + 1) * g]) * np.sign(blk) >= 0)


def test_quantize_exact_on_representable_rows():
    """A row whose values are E4M3 values times a power of two, with its largest
    magnitude 448 * 2^-7, quantizes to exactly those codes and dequantizes to x."""
    rng = np.random.default_rng(3)
    codes = rng.integers(0, 0x7F, (5, 128)).astype(np.uint8)
    codes[rng.random((5, 128)) < 0.5] |= 0x80
    codes[:, 7] = 0x7E
    x = om.e4m3_decode(codes) * 2.0 ** -7
    xb = oracle.f64_to_bf16(x)
    assert np.array_equal(oracle.bf16_to_f64(xb), x)
    q, s = oracle.quantize_fp8(xb, 128)
    assert np.all(s == 2.0 ** -7)
    assert np.array_equal(om.e4m3_decode(q), om.e4m3_decode(codes))
    assert np.array_equal(oracle.dequantize_fp8(q, s, 128), xb)


def test_dequantize_matches_library_steps():
    """decode -> fp32 multiply -> bf16, the same three steps through the library."""
    rng = np.random.default_rng(4)
    xb = _bf16_rows(rng, 17, 384, 3.0)
    for group in (0, 128):
        q, s = oracle.quantize_fp8(xb, group)
        g = 384 if group == 0 else 128
        qf = torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float32)
        sf = torch.from_numpy(s).repeat_interleave(g, dim=1)
        lib = (qf * sf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(oracle.dequantize_fp8(q, s, group), lib)
        # quantisation error of the round trip: half an E4M3 step of the group's scale
        err = np.abs(oracle.bf16_to_f64(oracle.dequantize_fp8(q, s, group)) - oracle.bf16_to_f64(xb))
        x = np.abs(oracle.bf16_to_f64(xb))
        smax = np.repeat(s.astype(np.float64), g, axis=1)
        assert np.all(err <= np.maximum(x * 2 ** -4, smax * 2 ** -10) * (1 + 2 ** -7) + x * 2 ** -8)


def test_scales_must_follow_the_row_permutation():
    """[M6.6] 0x0AC / 0x0AF: permuting the fp8 rows and their scales with the same
    map reproduces the dequantized token rows at every route row; scales left in
    token order give finite but wrong rows."""
    rng = np.random.default_rng(5)
    T, d, E, k = 12, 256, 4, 2
    xb = _bf16_rows(rng, T, d)
    xb = oracle.f64_to_bf16(oracle.bf16_to_f64(xb) * rng.uniform(0.1, 10, (T, 1)))
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)])
    p = oracle.permute(ids, E, -1)
    for group in (0, 128):
        q, s = oracle.quantize_fp8(xb, group)
        q_perm = oracle.gather_rows(q, p["row_to_route"], k)
        s_perm = oracle.gather_rows(s, p["row_to_route"], k)
        want = oracle.gather_rows(oracle.dequantize_fp8(q, s, group), p["row_to_route"], k)
        assert np.array_equal(oracle.dequantize_fp8(q_perm, s_perm, group), want)
        # the hazard: scales kept in route (token-major) order next to expert-major rows
        s_route_order = np.repeat(s, k, axis=0)[: q_perm.shape[0]]
        wrong = oracle.dequantize_fp8(q_perm, s_route_order, group)
        assert np.all(np.isfinite(oracle.bf16_to_f64(wrong)))
        assert not np.array_equal(wrong, want)
