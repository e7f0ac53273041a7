"""Per-kernel parity of the CUDA library against the CPU oracle, through the C
ABI, at sizes the oracle finishes in seconds: several tiles, ragged tails and
the degenerate cases (empty experts, capacity 0 and 1, T = 1, k = E, ties).
Integer outputs must match bit for bit; floats within the stated tolerances.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from moe_check import assert_float_parity, assert_gates, bits, host

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    from grouped_expert_gemm_gb300 import build
    build.build()
    torch.cuda.init()


def G():
    import grouped_expert_gemm_gb300 as g
    return g


def status0():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


# ----------------------------------------------------------------------------
# Router
# ----------------------------------------------------------------------------

def test_sigmoid_det_is_bitwise_identical_to_the_oracle():
    g = G()
    # every 13th fp32 bit pattern with |z| in [2^-24, 128), both signs, plus specials
    pos = np.arange(0x33800000, 0x43000000, 13, dtype=np.uint32)
    z = np.concatenate([pos.view(np.float32), -pos.view(np.float32),
                        np.array([0.0, -0.0, 87.0, -87.0, 88.0, -88.0, 1e30, -1e30, 3.4e38,
                                  -3.4e38], np.float32)])
    zd = torch.from_numpy(z).to(DEV)
    sd = torch.empty_like(zd)
    g.moe_sigmoid_det(z.size, zd, sd)
    torch.cuda.synchronize()
    got = host(sd).view(np.uint32)
    ref = oracle.sigmoid_det_f32(z).view(np.uint32)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, f"{bad.size} mismatches, first z={z[bad[:5]]}"


@pytest.mark.slow
def test_sigmoid_det_is_bitwise_identical_over_every_finite_fp32():
    """Every finite fp32 input (both signs, zeros, subnormals, |z| >= 128): the GPU's
    sigma_det and the oracle's give the same bits.  The oracle runs in chunks on a
    pool of spawned processes while the GPU works through the same chunks; each side
    reduces a chunk to a SHA-256 of its output bits, and a chunk whose digests differ
    is recomputed here to name its first differing inputs."""
    import hashlib
    import multiprocessing as mp
    import os

    import sigmoid_chunks as sc
    g = G()
    chunks = sc.finite_chunks()
    assert sum(n for _, n in chunks) == 2 * 0x7F800000
    ctx = mp.get_context("spawn")
    with ctx.Pool(max(1, min(16, os.cpu_count() or 1))) as pool:
        pending = pool.starmap_async(sc.oracle_chunk_digest, chunks)
        gpu = []
        zd = torch.empty(sc.CHUNK, dtype=torch.int32, device=DEV)
        sd = torch.empty(sc.CHUNK, dtype=torch.float32, device=DEV)
        for start, n in chunks:
            signed = start - (1 << 32) if start >= (1 << 31) else start
            torch.arange(signed, signed + n, dtype=torch.int32, device=DEV, out=zd[:n])
            g.moe_sigmoid_det(n, zd[:n].view(torch.float32), sd[:n])
            gpu.append(hashlib.sha256(host(sd[:n]).view(np.uint8)).hexdigest())
        ref = pending.get(timeout=1800)
    bad = [i for i, (a, b) in enumerate(zip(gpu, ref)) if a != b]
    if bad:
        start, n = chunks[bad[0]]
        signed = start - (1 << 32) if start >= (1 << 31) else start
        torch.arange(signed, signed + n, dtype=torch.int32, device=DEV, out=zd[:n])
        g.moe_sigmoid_det(n, zd[:n].view(torch.float32), sd[:n])
        got = host(sd[:n]).view(np.uint32)
        want = sc.oracle_chunk(start, n).view(np.uint32)
        where = np.nonzero(got != want)[0][:5]
        raise AssertionError(f"{len(bad)} chunks differ; first inputs (bits) "
                             f"{[hex(start + int(i)) for i in where]}")


def _route(w, logits, sel_bias):
    g = G()
    score = g.MOE_SCORE_SOFTMAX if w.score_fn == "softmax" else g.MOE_SCORE_SIGMOID_GROUP
    p = g.RouteParams(w.T, w.E, w.k, score, w.n_group, w.topk_group, w.route_scale)
    ids = torch.empty((w.T, w.k), dtype=torch.int32, device=DEV)
    gates = torch.empty((w.T, w.k), dtype=torch.float32, device=DEV)
    st = status0()
    g.moe_route(p, logits, sel_bias, ids, gates, st)
    torch.cuda.synchronize()
    return host(ids), host(gates), int(host(st)[0])


@pytest.mark.parametrize("T,E,k", [(1, 8, 2), (257, 8, 2), (300, 128, 8), (77, 384, 8),
                                   (64, 512, 16), (33, 5, 5), (40, 33, 3), (19, 1, 1)])
def test_route_softmax_parity(T, E, k):
    w = workloads.scaled(workloads.tiny(), T=T, E=E, k=k)
    logits, _ = workloads.make_router_inputs(w, DEV)
    ids, gates, st = _route(w, logits, None)
    rids, rgates = oracle.route_softmax(host(logits), k)
    assert st == 0
    assert np.array_equal(ids, rids)
    assert_gates(gates, rgates)


def test_route_softmax_ties_and_signed_zeros():
    rng = np.random.default_rng(0)
    z = rng.choice(np.array([-1.0, -0.0, 0.0, 0.5, 2.0], np.float32), size=(512, 40))
    w = workloads.scaled(workloads.tiny(), T=512, E=40, k=6)
    ids, gates, _ = _route(w, torch.from_numpy(z).to(DEV), None)
    rids, rgates = oracle.route_softmax(z, 6)
    assert np.array_equal(ids, rids)
    assert_gates(gates, rgates)


def test_route_nan_logit_is_reported_and_ranked_last():
    z = np.zeros((4, 8), np.float32)
    z[:, 3] = 1.0
    z[1, 5] = np.nan
    w = workloads.scaled(workloads.tiny(), T=4, E=8, k=2)
    ids, _, st = _route(w, torch.from_numpy(z).to(DEV), None)
    g = G()
    assert st & g.MOE_DEV_NONFINITE_LOGIT
    assert ids[1].tolist() == [3, 0]


@pytest.mark.parametrize("T,E,n_group,topk_group,k", [(1, 256, 8, 4, 8), (513, 256, 8, 4, 8),
                                                      (100, 64, 4, 2, 6), (50, 12, 4, 2, 4)])
def test_route_sigmoid_group_parity(T, E, n_group, topk_group, k):
    w = workloads.scaled(workloads.v3(), T=T, E=E, k=k, n_group=n_group, topk_group=topk_group)
    logits, sel_bias = workloads.make_router_inputs(w, DEV)
    ids, gates, st = _route(w, logits, sel_bias)
    rids, rgates = oracle.route_sigmoid_group(host(logits), host(sel_bias), k, n_group,
                                              topk_group, 2.5)
    assert st == 0
    assert np.array_equal(ids, rids)
    assert_gates(gates, rgates)


def test_route_sigmoid_group_page_fixture():
    import json, os
    with open(os.path.join(os.path.dirname(__file__), "golden", "m62_v3_group_gate.json")) as f:
        fx = json.load(f)
    p = np.asarray(fx["affinity"], np.float64)
    z = np.float32(np.log(p / (1 - p)))[None, :]
    w = workloads.scaled(workloads.v3(), T=1, E=12, k=4, n_group=4, topk_group=2)
    ids, gates, _ = _route(w, torch.from_numpy(z).to(DEV),
                           torch.tensor(fx["bias"], dtype=torch.float32, device=DEV))
    assert ids[0].tolist() == fx["ids_with_bias"]
    np.testing.assert_allclose(gates[0], fx["gates_with_bias"], atol=1.5e-6)


# ----------------------------------------------------------------------------
# Permute
# ----------------------------------------------------------------------------

def _permute(T, d, E, k, cap, ids_np, x):
    g = G()
    R = T * k
    ids = torch.from_numpy(np.ascontiguousarray(ids_np, dtype=np.int32)).to(DEV)
    xp = torch.full((max(R, 1), d), -1, dtype=torch.bfloat16, device=DEV)
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    r2r = torch.full((max(R, 1),), -7, dtype=torch.int32, device=DEV)
    inv = torch.full((max(R, 1),), -7, dtype=torch.int32, device=DEV)
    nd = torch.zeros(1, dtype=torch.int32, device=DEV)
    wsb = g.moe_permute_workspace_size(T, k, E)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    st = status0()
    g.moe_permute(T, d, E, k, cap, ids, x, xp, counts, offsets, r2r, inv, nd, ws, wsb, st)
    torch.cuda.synchronize()
    return dict(x_perm=bits(xp), counts=host(counts), offsets=host(offsets),
                row_to_route=host(r2r), route_to_row=host(inv), n_dropped=int(host(nd)[0]),
                status=int(host(st)[0]))


def _check_permute(T, d, E, k, cap, ids_np, seed=0):
    gen = torch.Generator(device=DEV).manual_seed(seed)
    x = torch.randn((max(T, 1), d), generator=gen, device=DEV).to(torch.bfloat16)[:T]
    got = _permute(T, d, E, k, cap, ids_np, x)
    ref = oracle.permute(ids_np, E, cap)
    acc = int(ref["offsets"][-1])
    assert got["status"] == 0
    assert np.array_equal(got["counts"], ref["counts"])
    assert np.array_equal(got["offsets"], ref["offsets"])
    assert np.array_equal(got["row_to_route"][:acc], ref["row_to_route"])
    assert np.array_equal(got["route_to_row"][:T * k], ref["route_to_row"])
    assert got["n_dropped"] == ref["n_dropped"]
    xb = bits(x)
    assert np.array_equal(got["x_perm"][:acc], oracle.gather_rows(xb, ref["row_to_route"], k))


@pytest.mark.parametrize("T,d,E,k,cap", [(256, 64, 8, 2, 80), (1, 64, 8, 2, -1), (3, 64, 8, 8, -1),
                                         (1000, 128, 128, 8, -1), (997, 64, 256, 8, 31),
                                         (4099, 64, 8, 2, 0), (500, 64, 16, 4, 1),
                                         (129, 192, 384, 8, -1), (2000, 64, 512, 16, 40),
                                         (64, 64, 1, 1, -1), (2, 4096, 16, 8, 1)])
def test_permute_parity(T, d, E, k, cap):
    rng = np.random.default_rng(T + E)
    # skewed expert choice so that some experts are empty and some overflow
    p = rng.dirichlet(np.ones(E) * 0.3)
    ids = np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    _check_permute(T, d, E, k, cap, ids)


def test_permute_empty_input():
    got = _permute(0, 64, 8, 2, -1, np.zeros((0, 2), np.int32),
                   torch.empty((0, 64), dtype=torch.bfloat16, device=DEV))
    assert got["counts"].tolist() == [0] * 8
    assert got["offsets"].tolist() == [0] * 9
    assert got["n_dropped"] == 0


def test_permute_bad_expert_id_is_reported_and_dropped():
    ids = np.array([[0, 1], [9, 2], [1, -3]], np.int32)
    x = torch.zeros((3, 64), dtype=torch.bfloat16, device=DEV)
    got = _permute(3, 64, 4, 2, -1, ids, x)
    g = G()
    assert got["status"] & g.MOE_DEV_BAD_EXPERT_ID
    assert got["route_to_row"][2] == -1 and got["route_to_row"][5] == -1
    assert got["counts"].tolist() == [1, 2, 1, 0]
    assert got["n_dropped"] == 2


# ----------------------------------------------------------------------------
# Combine
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("T,k,d,rows,shared,accumulate", [(256, 2, 64, 400, False, False),
                                                          (33, 8, 2048, 200, True, False),
                                                          (100, 16, 1032, 999, False, True),
                                                          (1, 1, 8, 1, True, True)])
def test_combine_parity(T, k, d, rows, shared, accumulate):
    g = G()
    rng = np.random.default_rng(T * k)
    gen = torch.Generator(device=DEV).manual_seed(1)
    y = torch.randn((rows, d), generator=gen, device=DEV).to(torch.bfloat16)
    r2r = rng.integers(-1, rows, size=T * k).astype(np.int32)
    gates = rng.uniform(0, 1, size=T * k).astype(np.float32)
    sh = torch.randn((T, d), generator=gen, device=DEV).to(torch.bfloat16) if shared else None
    init = torch.randn((T, d), generator=gen, device=DEV, dtype=torch.float32)
    out = init.clone()
    st = status0()
    g.moe_combine(T, k, d, y, rows, torch.from_numpy(r2r).to(DEV), torch.from_numpy(gates).to(DEV),
                  sh, accumulate, out, st)
    torch.cuda.synchronize()
    ref = oracle.combine(oracle.bf16_to_f64(bits(y)), r2r, gates, T, k,
                         None if sh is None else oracle.bf16_to_f64(bits(sh)),
                         host(init) if accumulate else None)
    assert int(host(st)[0]) == 0
    assert_float_parity(host(out), ref, "combine")
    # fp32 accumulation of at most k+2 terms: far inside the bar
    np.testing.assert_allclose(host(out), ref, rtol=1e-5, atol=1e-5)


def test_combine_bad_row_is_reported_and_skipped():
    g = G()
    y = torch.ones((4, 8), dtype=torch.bfloat16, device=DEV)
    r2r = torch.tensor([0, 7], dtype=torch.int32, device=DEV)
    gates = torch.tensor([0.5, 0.5], dtype=torch.float32, device=DEV)
    out = torch.empty((1, 8), dtype=torch.float32, device=DEV)
    st = status0()
    g.moe_combine(1, 2, 8, y, 4, r2r, gates, None, 0, out, st)
    torch.cuda.synchronize()
    assert int(host(st)[0]) & g.MOE_DEV_BAD_ROW
    assert np.allclose(host(out), 0.5)


# ----------------------------------------------------------------------------
# Grouped SwiGLU GEMM
# ----------------------------------------------------------------------------

def _gemm_case(n_seg, d, I, counts, begins=None, seed=0, max_rows=None, sample=None):
    g = G()
    counts = np.asarray(counts, np.int32)
    if begins is None:
        begins = np.concatenate([[0], np.cumsum(counts)[:-1]]).astype(np.int32)
    begins = np.asarray(begins, np.int32)
    if max_rows is None:
        max_rows = int((begins + counts).max()) if len(counts) else 1
    w = workloads.scaled(workloads.tiny(), d=d, I=I, E=n_seg, seed=seed)
    gen = torch.Generator(device=DEV).manual_seed(seed + 7)
    x = torch.randn((max_rows, d), generator=gen, device=DEV).to(torch.bfloat16)
    wg, wu, wd = workloads.make_expert_weights(w, DEV, n_experts=n_seg)
    y = torch.full((max_rows, d), 7.0, dtype=torch.bfloat16, device=DEV)
    wsb = g.moe_grouped_swiglu_workspace_size(max_rows, I)
    ws = torch.zeros(wsb, dtype=torch.uint8, device=DEV)
    st = status0()
    g.moe_grouped_swiglu(n_seg, d, I, max_rows, x, torch.from_numpy(begins).to(DEV),
                         torch.from_numpy(counts).to(DEV), wg, wu, wd, y, ws, wsb, st)
    torch.cuda.synchronize()
    assert int(host(st)[0]) == 0
    H = ws[: max_rows * I * 2].view(torch.bfloat16).view(max_rows, I)
    pick = None
    if sample is not None:
        all_rows = np.concatenate([np.arange(b, b + c) for b, c in zip(begins, counts)])
        pick = np.sort(np.random.default_rng(seed).choice(all_rows, sample, replace=False))
    yr, hr = oracle.grouped_swiglu_rows(bits(x), begins, counts, bits(wg), bits(wu), bits(wd),
                                        rows=pick)
    rows = sorted(yr)
    yb, hb = bits(y), bits(H)
    if rows:
        assert_float_parity(oracle.bf16_to_f64(hb[rows]),
                            oracle.bf16_to_f64(np.stack([hr[r] for r in rows])), "H")
        assert_float_parity(oracle.bf16_to_f64(yb[rows]),
                            oracle.bf16_to_f64(np.stack([yr[r] for r in rows])), "y")
    # rows outside every segment are never written
    seg_rows = np.concatenate([np.arange(b, b + c) for b, c in zip(begins, counts)]) \
        if len(counts) else np.zeros(0, int)
    untouched = np.setdiff1d(np.arange(max_rows), seg_rows)
    assert np.all(yb[untouched] == bits(torch.tensor([7.0], dtype=torch.bfloat16))[0])


@pytest.mark.parametrize("n_seg,d,I,counts", [
    (1, 64, 128, [128]),
    (1, 64, 128, [1]),
    (4, 64, 128, [130, 0, 7, 300]),
    (3, 128, 256, [255, 256, 257]),
    (5, 256, 384, [1, 129, 0, 64, 200]),
    (8, 512, 128, [33, 97, 128, 5, 0, 0, 140, 61]),
    (2, 192, 192, [150, 170]),       # I not a multiple of 128, d not of 256
    (6, 1024, 512, [400, 10, 300, 0, 129, 77]),
])
def test_grouped_swiglu_parity(n_seg, d, I, counts):
    _gemm_case(n_seg, d, I, counts)


@pytest.mark.parametrize("d,I", [(4096, 256), (256, 8192)])
def test_grouped_swiglu_large_segments_row_block_outer_order(d, I):
    # Segments of ~8 K rows whose A does not fit the L2 budget while one expert's
    # weights do: the gate/up pass (d=4096) or the down pass (I=8192) then walks
    # each block of rows across all weight columns before the next block.
    _gemm_case(2, d, I, [8191, 8193], sample=300)


def test_grouped_swiglu_many_experts_few_rows():
    # decode-like: 64 experts of a few rows each (single-CTA kernel, 2x128 gate/up tiles)
    rng = np.random.default_rng(21)
    _gemm_case(64, 128, 768, rng.integers(0, 20, size=64))


def test_grouped_swiglu_gapped_segments():
    # segments with gaps between them (the pooled layout's fixed-stride arrays)
    _gemm_case(3, 128, 128, [100, 0, 250], begins=[0, 300, 600], max_rows=900)


def test_grouped_swiglu_many_small_segments():
    rng = np.random.default_rng(3)
    counts = rng.integers(0, 40, size=256)
    _gemm_case(256, 64, 128, counts)


def test_grouped_swiglu_max_segments():
    """1024 segments, the limit: the device segment table (8 segments per thread) and
    the tile scheduler over many empty and tiny segments."""
    rng = np.random.default_rng(1024)
    _gemm_case(1024, 64, 128, rng.integers(0, 4, size=1024), sample=256)


_R5 = np.random.default_rng(5)
DEEP_CASES = [
    # (n_seg, d, I, counts): narrow tiles with at most 32 rows per box and K a multiple
    # of 128, so both passes run 128-K stages of 128-row weight boxes
    (128, 2048, 768, [1 if e % 16 == 3 else 0 for e in range(128)]),  # one-token decode
    (32, 256, 768, list(_R5.integers(1, 4, size=32))),     # gate/up: 384 tiles, ring wraps
    (24, 2048, 256, list(_R5.integers(1, 5, size=24))),    # down: 384 tiles, 2 k-steps
    (16, 384, 384, [7, 0, 8, 5, 6, 8, 8, 1, 0, 7, 3, 8, 40, 6, 2, 8]),  # 32-row boxes, ragged
]


@pytest.mark.parametrize("n_seg,d,I,counts", DEEP_CASES)
def test_grouped_swiglu_deep_stages(n_seg, d, I, counts):
    """Decode-sized segments on the single-CTA kernel's 128-K stages (two A boxes and
    one 128-row box per weight atom per stage) against the oracle, every row."""
    _gemm_case(n_seg, d, I, counts)


@pytest.mark.parametrize("n_seg,d,I,counts", [
    (128, 2048, 768, [1 if e % 16 == 3 else 0 for e in range(128)]),  # one-token decode, 128-K stages
    DEEP_CASES[2],                                  # 128-K stages, several down tiles per CTA
    (8, 192, 128, [3, 0, 5, 1, 0, 2, 7, 4]),       # one 64-column atom, 2 k-steps < ring depth
    (4, 128, 256, [40, 0, 17, 90]),                 # two atoms, 64-row boxes
    (64, 512, 1024, [30 + (e * 7) % 11 for e in range(64)]),  # several tiles per CTA
    (2, 256, 128, [300, 260]),                      # CTA-pair kernel (chaining not used)
])
def test_down_chained_equals_plain_down(n_seg, d, I, counts):
    """The chained down pass (weights staged before the gate/up pass ends) writes the
    same y bits as the plain call, on every kernel shape; sampled rows match the oracle."""
    g = G()
    counts = np.asarray(counts, np.int32)
    begins = np.concatenate([[0], np.cumsum(counts)[:-1]]).astype(np.int32)
    max_rows = max(int(counts.sum()), 1)
    w = workloads.scaled(workloads.tiny(), d=d, I=I, E=n_seg, seed=5)
    gen = torch.Generator(device=DEV).manual_seed(12)
    x = torch.randn((max_rows, d), generator=gen, device=DEV).to(torch.bfloat16)
    wg, wu, wd = workloads.make_expert_weights(w, DEV, n_experts=n_seg)
    b_t, c_t = torch.from_numpy(begins).to(DEV), torch.from_numpy(counts).to(DEV)
    h = torch.empty((max_rows, I), dtype=torch.bfloat16, device=DEV)
    ys = []
    st = status0()
    for chained in (False, True):
        y = torch.full((max_rows, d), 7.0, dtype=torch.bfloat16, device=DEV)
        g.moe_grouped_gate_up(n_seg, d, I, max_rows, x, b_t, c_t, wg, wu, h, st)
        down = g.moe_grouped_down_chained if chained else g.moe_grouped_down
        down(n_seg, I, d, max_rows, h, b_t, c_t, wd, y, st)
        ys.append(y)
    torch.cuda.synchronize()
    assert int(host(st)[0]) == 0
    assert np.array_equal(bits(ys[0]), bits(ys[1]))
    pick = np.sort(np.random.default_rng(3).choice(int(counts.sum()), min(8, int(counts.sum())),
                                                   replace=False))
    yr, _ = oracle.grouped_swiglu_rows(bits(x), begins, counts, bits(wg), bits(wu), bits(wd),
                                       rows=pick)
    r = sorted(yr)
    assert_float_parity(oracle.bf16_to_f64(bits(ys[1])[r]),
                        oracle.bf16_to_f64(np.stack([yr[i] for i in r])), "y")


def test_grouped_swiglu_bad_segment_is_reported():
    g = G()
    d, I = 64, 128
    x = torch.zeros((16, d), dtype=torch.bfloat16, device=DEV)
    w = torch.zeros((1, d, I), dtype=torch.bfloat16, device=DEV)
    wd = torch.zeros((1, I, d), dtype=torch.bfloat16, device=DEV)
    y = torch.zeros((16, d), dtype=torch.bfloat16, device=DEV)
    wsb = g.moe_grouped_swiglu_workspace_size(16, I)
    ws = torch.zeros(wsb, dtype=torch.uint8, device=DEV)
    st = status0()
    g.moe_grouped_swiglu(1, d, I, 16, x, torch.tensor([10], dtype=torch.int32, device=DEV),
                         torch.tensor([20], dtype=torch.int32, device=DEV), w, w, wd, y, ws, wsb, st)
    torch.cuda.synchronize()
    assert int(host(st)[0]) & g.MOE_DEV_BAD_ROW


def _gather_case(T, d, E, k, I, cap=-1, seed=0, alpha=1.0):
    """gate/up with rows gathered from token order vs the same pass on moe_permute's
    copy: H bit-identical on every segment row, other rows untouched."""
    g = G()
    rng = np.random.default_rng(seed)
    p = rng.dirichlet(np.ones(E) * alpha)
    ids_np = np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    gen = torch.Generator(device=DEV).manual_seed(seed + 1)
    x = torch.randn((T, d), generator=gen, device=DEV).to(torch.bfloat16)
    w = workloads.scaled(workloads.tiny(), d=d, I=I, E=E, seed=seed)
    wg, wu, _ = workloads.make_expert_weights(w, DEV, n_experts=E)
    R = T * k
    got = _permute(T, d, E, k, cap, ids_np, x)  # maps and the copied rows
    i32 = dict(dtype=torch.int32, device=DEV)
    counts, offsets = torch.from_numpy(got["counts"]).to(DEV), torch.from_numpy(got["offsets"]).to(DEV)
    r2r = torch.from_numpy(got["row_to_route"]).to(DEV)
    xp = torch.from_numpy(got["x_perm"].view(np.int16)).to(DEV).view(torch.bfloat16)
    h_copy = torch.full((R, I), 3.0, dtype=torch.bfloat16, device=DEV)
    h_gath = torch.full((R, I), 3.0, dtype=torch.bfloat16, device=DEV)
    st = status0()
    g.moe_grouped_gate_up(E, d, I, R, xp, offsets, counts, wg, wu, h_copy, st)
    g.moe_grouped_gate_up_gather(E, d, I, R, T, k, x, r2r, offsets, counts, wg, wu, h_gath, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(h_copy.view(torch.int16), h_gath.view(torch.int16))
    acc = int(got["offsets"][-1])
    assert torch.all(h_gath[acc:] == 3.0)
    # and H against the oracle on a few rows
    if acc:
        rows = np.sort(rng.choice(acc, min(acc, 24), replace=False))
        xb = bits(x)
        for r in rows:
            e = int(np.searchsorted(got["offsets"], r, side="right") - 1)
            xr = oracle.bf16_to_f64(xb[got["row_to_route"][r] // k][None])
            gg = xr @ oracle.bf16_to_f64(bits(wg[e]))
            uu = xr @ oracle.bf16_to_f64(bits(wu[e]))
            ref = oracle.bf16_to_f64(oracle.f64_to_bf16(oracle.silu(gg) * uu))
            assert_float_parity(oracle.bf16_to_f64(bits(h_gath[r:r + 1])), ref, f"H row {r}")


@pytest.mark.parametrize("T,d,E,k,I,cap", [
    (1, 2048, 128, 8, 768, -1),    # one token: 16-row boxes, 2 x 64-column tiles
    (8, 2048, 128, 8, 768, -1),
    (128, 256, 128, 8, 768, -1),   # decode T=128 shape class: 32-row boxes, wide tiles
    (300, 256, 32, 4, 192, -1),    # I not a multiple of 128
    (1000, 128, 8, 2, 256, 200),   # capacity with drops
    (4096, 512, 8, 2, 256, -1),    # CTA-pair kernel (segments average >= 128 rows)
    (2000, 256, 16, 4, 384, 480),  # pair kernel with ragged tails and drops
])
def test_gate_up_gather_equals_copy_path(T, d, E, k, I, cap):
    _gather_case(T, d, E, k, I, cap, seed=T + E)


@pytest.mark.parametrize("T,E,k,cap", [(300, 32, 4, 40), (5000, 128, 8, -1), (1, 8, 2, -1)])
def test_permute_maps_only_equals_the_copying_call(T, E, k, cap):
    """x = x_perm = NULL: the same maps, counts, offsets and drops, and one launch fewer
    where the rows have a copy launch of their own (above 16 routes)."""
    g = G()
    rng = np.random.default_rng(T)
    ids_np = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    x = torch.randn((T, 64), device=DEV).to(torch.bfloat16)
    full = _permute(T, 64, E, k, cap, ids_np, x)
    ids = torch.from_numpy(ids_np).to(DEV)
    i32 = dict(dtype=torch.int32, device=DEV)
    counts, offsets = torch.empty(E, **i32), torch.empty(E + 1, **i32)
    r2r, inv = torch.full((T * k,), -7, **i32), torch.full((T * k,), -7, **i32)
    nd = torch.zeros(1, **i32)
    wsb = g.moe_permute_workspace_size(T, k, E)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    st = status0()
    n0 = g.launch_count()
    g.moe_permute(T, 64, E, k, cap, ids, None, None, counts, offsets, r2r, inv, nd, ws, wsb, st)
    assert g.launch_count() - n0 == g.abi._permute_launches(T, k, copy=False)
    assert g.abi._permute_launches(T, k, copy=False) == \
        g.abi._permute_launches(T, k) - (1 if T * k > 16 else 0)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    acc = int(full["offsets"][-1])
    assert np.array_equal(host(counts), full["counts"])
    assert np.array_equal(host(offsets), full["offsets"])
    assert np.array_equal(host(r2r)[:acc], full["row_to_route"][:acc])
    assert np.array_equal(host(inv), full["route_to_row"][:T * k])
    assert int(nd.item()) == full["n_dropped"]


def test_gate_up_gather_bad_map_entry_is_reported():
    g = G()
    T, d, E, k, I = 16, 64, 4, 2, 128
    x = torch.randn((T, d), device=DEV).to(torch.bfloat16)
    wg = torch.zeros((E, d, I), dtype=torch.bfloat16, device=DEV)
    r2r = torch.arange(T * k, dtype=torch.int32, device=DEV)
    r2r[5] = T * k + 3  # outside the routes
    counts = torch.full((E,), T * k // E, dtype=torch.int32, device=DEV)
    offsets = torch.arange(E + 1, dtype=torch.int32, device=DEV) * (T * k // E)
    h = torch.zeros((T * k, I), dtype=torch.bfloat16, device=DEV)
    st = status0()
    g.moe_grouped_gate_up_gather(E, d, I, T * k, T, k, x, r2r, offsets, counts, wg, wg, h, st)
    torch.cuda.synchronize()
    assert int(st.item()) & g.MOE_DEV_BAD_ROW


# ----------------------------------------------------------------------------
# Pooled layout
# ----------------------------------------------------------------------------

def _pool_case(T, d, k, n_dest, L, n_waves, pool_cap, local_cap, policy, seed=0):
    g = G()
    rng = np.random.default_rng(seed)
    E = n_dest * L
    p = rng.dirichlet(np.ones(E) * 0.5)
    ids_np = np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    gen = torch.Generator(device=DEV).manual_seed(seed)
    x = torch.randn((T, d), generator=gen, device=DEV).to(torch.bfloat16)
    xb = bits(x)
    ids = torch.from_numpy(ids_np).to(DEV)
    pp = g.PoolParams(n_dest, L, n_waves, pool_cap, policy)
    pols = {g.MOE_WAVE_STRIPE: "stripe", g.MOE_WAVE_DESTMOD: "destmod"}
    pools = torch.zeros((n_dest, pool_cap + 1, d), dtype=torch.bfloat16, device=DEV)
    r2p = torch.empty(T * k, dtype=torch.int32, device=DEV)
    fill = torch.empty(n_dest, dtype=torch.int32, device=DEV)
    sdrop = torch.zeros(1, dtype=torch.int32, device=DEV)
    pwsb = g.moe_pool_pack_workspace_size(pp, T, k)
    pws = torch.empty(pwsb, dtype=torch.uint8, device=DEV)
    compact = torch.zeros((L * local_cap, d), dtype=torch.bfloat16, device=DEV)
    lcounts = torch.empty(L, dtype=torch.int32, device=DEV)
    p2r = torch.empty(n_dest * pool_cap, dtype=torch.int32, device=DEV)
    rdrop = torch.zeros(1, dtype=torch.int32, device=DEV)
    cwsb = g.moe_pool_compact_workspace_size(n_dest, pool_cap, L)
    cws = torch.empty(cwsb, dtype=torch.uint8, device=DEV)
    comp = torch.empty(T * k, dtype=torch.int32, device=DEV)
    total = 0
    for wave in range(n_waves):
        st = status0()
        g.moe_pool_pack(pp, T, d, k, wave, ids, x, pools, r2p, fill, sdrop, pws, pwsb, st)
        g.moe_pool_compact(n_dest, pool_cap, d, L, local_cap, pools, compact, lcounts, p2r, rdrop,
                           cws, cwsb, st)
        g.moe_compose_map(T * k, r2p, p2r, n_dest * pool_cap, comp, st)
        torch.cuda.synchronize()
        assert int(host(st)[0]) == 0
        rp = oracle.pool_pack(ids_np, xb, n_dest, L, n_waves, pool_cap, wave, pols[policy])
        pb = bits(pools)
        assert np.array_equal(pb[:, 0, :], rp["pools"][:, 0, :])  # whole header rows
        assert np.array_equal(host(r2p), rp["route_to_poolrow"])
        assert np.array_equal(host(fill), rp["fill"])
        assert int(host(sdrop)[0]) == rp["sender_drops"]
        for D in range(n_dest):
            f = rp["fill"][D]
            assert np.array_equal(pb[D, 1:1 + f], rp["pools"][D, 1:1 + f])
        rc = oracle.pool_compact(rp["pools"], pool_cap, L, local_cap)
        assert np.array_equal(host(p2r), rc["poolrow_to_row"])
        assert np.array_equal(host(lcounts), rc["local_counts"])
        assert int(host(rdrop)[0]) == rc["receiver_drops"]
        cb = bits(compact).reshape(L, local_cap, d)
        for l in range(L):
            c = rc["local_counts"][l]
            assert np.array_equal(cb[l, :c], rc["compact"][l, :c])
        rcomp = oracle.compose_map(rp["route_to_poolrow"], rc["poolrow_to_row"])
        assert np.array_equal(host(comp), rcomp)
        total += rp["sender_drops"] + rc["receiver_drops"] + int((rcomp >= 0).sum())
    assert total == T * k


@pytest.mark.parametrize("policy", [0, 1])
@pytest.mark.parametrize("T,d,k,n_dest,L,n_waves,pool_cap,local_cap", [
    (300, 64, 4, 4, 3, 3, 40, 50),
    (1000, 128, 8, 16, 6, 3, 64, 150),
    (77, 64, 2, 2, 2, 1, 64, 1000),     # nothing dropped
    (500, 64, 8, 8, 4, 2, 5, 7),        # heavy drops on both sides
    (3, 64, 2, 16, 2, 2, 8, 4),         # most pools (and local experts) empty
])
def test_pool_pack_compact_parity(policy, T, d, k, n_dest, L, n_waves, pool_cap, local_cap):
    _pool_case(T, d, k, n_dest, L, n_waves, pool_cap, local_cap, policy)


@pytest.mark.parametrize("first", [1, 5, 7])
def test_pool_compact_rotated_parity(first):
    """The per-receiver rotation of the source order: same maps, counts and drops as the
    oracle visiting sources from `first` on; the overflow falls on other sources."""
    g = G()
    T, d, k, n_dest, L, pool_cap, local_cap = 600, 64, 4, 8, 3, 40, 40
    rng = np.random.default_rng(first)
    E = n_dest * L
    p = rng.dirichlet(np.ones(E) * 0.5)
    ids_np = np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    x = torch.randn((T, d), device=DEV).to(torch.bfloat16)
    pp = g.PoolParams(n_dest, L, 1, pool_cap, g.MOE_WAVE_STRIPE)
    pools = torch.zeros((n_dest, pool_cap + 1, d), dtype=torch.bfloat16, device=DEV)
    i32 = dict(dtype=torch.int32, device=DEV)
    r2p, fill, sdrop = torch.empty(T * k, **i32), torch.empty(n_dest, **i32), torch.zeros(1, **i32)
    pwsb = g.moe_pool_pack_workspace_size(pp, T, k)
    pws = torch.empty(pwsb, dtype=torch.uint8, device=DEV)
    st = status0()
    g.moe_pool_pack(pp, T, d, k, 0, torch.from_numpy(ids_np).to(DEV), x, pools, r2p, fill, sdrop,
                    pws, pwsb, st)
    compact = torch.zeros((L * local_cap, d), dtype=torch.bfloat16, device=DEV)
    lcounts, p2r, rdrop = torch.empty(L, **i32), torch.empty(n_dest * pool_cap, **i32), torch.zeros(1, **i32)
    cwsb = g.moe_pool_compact_workspace_size(n_dest, pool_cap, L)
    cws = torch.empty(cwsb, dtype=torch.uint8, device=DEV)
    g.moe_pool_compact_rotated(n_dest, pool_cap, d, L, local_cap, first, pools, compact, lcounts,
                               p2r, rdrop, cws, cwsb, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    pb = bits(pools)
    rc = oracle.pool_compact(pb, pool_cap, L, local_cap, first)
    assert rc["receiver_drops"] > 0  # the case overflows
    assert np.array_equal(host(p2r), rc["poolrow_to_row"])
    assert np.array_equal(host(lcounts), rc["local_counts"])
    assert int(rdrop.item()) == rc["receiver_drops"]
    cb = bits(compact).reshape(L, local_cap, d)
    for l in range(L):
        c = int(rc["local_counts"][l])
        assert np.array_equal(cb[l, :c], rc["compact"][l, :c])
    base = oracle.pool_compact(pb, pool_cap, L, local_cap)
    assert not np.array_equal(base["poolrow_to_row"], rc["poolrow_to_row"])


def test_pool_compact_bad_header_is_reported():
    g = G()
    d, cap = 16, 4
    pools = torch.full((2, cap + 1, d), 0, dtype=torch.int16, device=DEV)
    hdr = np.full((2, d), 0xFFFF, np.uint16)
    hdr[0, :3] = [0, 9, 1]
    pools[:, 0, :] = torch.from_numpy(hdr.view(np.int16)).to(DEV)
    pools = pools.view(torch.bfloat16)
    compact = torch.zeros((2 * 8, d), dtype=torch.bfloat16, device=DEV)
    lc = torch.empty(2, dtype=torch.int32, device=DEV)
    p2r = torch.empty(2 * cap, dtype=torch.int32, device=DEV)
    rd = torch.zeros(1, dtype=torch.int32, device=DEV)
    wsb = g.moe_pool_compact_workspace_size(2, cap, 2)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    st = status0()
    g.moe_pool_compact(2, cap, d, 2, 8, pools, compact, lc, p2r, rd, ws, wsb, st)
    torch.cuda.synchronize()
    assert int(host(st)[0]) & g.MOE_DEV_BAD_HEADER_ID
    assert host(p2r).tolist() == [0, -1, 8, -1, -1, -1, -1, -1]
