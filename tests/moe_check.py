"""Helpers shared by the GPU parity tests: tolerance checks and the oracle's
pipeline on host copies of the inputs the CUDA path received."""
import json
import os

import numpy as np
import torch

import oracle
import workloads

# Floating-point parity bar.  The stated bar pairs a maximum relative error with
# a normwise one; they are read as the relative error in the max norm and in the
# 2-norm:
#   max_rel  = ||x - r||_inf / ||r||_inf   <= 1e-2
#   normwise = ||x - r||_2   / ||r||_2     <= 2e-3
# and every element must also satisfy an element-wise bound derived from the
# arithmetic: |x_i - r_i| <= 2^-6 * max(|r_i|, rms(r)).  The outputs pass through
# two bf16 roundings (H, then y) on top of fp32 accumulation in the tensor cores
# (fp64 in the oracle).  Where the fp32 and fp64 sums straddle a bf16 rounding
# boundary the two sides round to neighbouring values, one bf16 ulp apart: at
# most 2^-7 relative for y, and an H value off by one ulp feeds a further error of
# the same order into y.  Two bf16 ulps, 2^-6, bound both; the rms floor keeps the
# bound meaningful for elements near zero, whose relative error is undefined.
MAX_REL = 1e-2
NORMWISE = 2e-3
ELEMENT = 2.0 ** -6
# Gates are fp32 results of a few fp32 operations: relative 2e-6 plus 1e-7 absolute.
GATE_RTOL, GATE_ATOL = 2e-6, 1e-7

# With MOE_PARITY_LOG=<path>, every float parity check appends its three measured
# errors to that file as one JSON line (the record of the observed maxima).
PARITY_LOG = os.environ.get("MOE_PARITY_LOG")


def float_errors(got, ref):
    """(max-norm relative, 2-norm relative, element-wise with rms floor) errors."""
    got = np.asarray(got, dtype=np.float64).ravel()
    ref = np.asarray(ref, dtype=np.float64).ravel()
    if ref.size == 0:
        return 0.0, 0.0, 0.0
    diff = np.abs(got - ref)
    rinf = float(np.max(np.abs(ref)))
    max_rel = float(diff.max() / (rinf if rinf > 0 else 1.0))
    nref = float(np.linalg.norm(ref))
    normwise = float(np.linalg.norm(got - ref) / (nref if nref > 0 else 1.0))
    rms = float(np.sqrt(np.mean(ref * ref)))
    elem = float(np.max(diff / np.maximum(np.abs(ref), rms if rms > 0 else 1.0)))
    return max_rel, normwise, elem


def assert_float_parity(got, ref, what=""):
    mr, nw, el = float_errors(got, ref)
    if PARITY_LOG:
        with open(PARITY_LOG, "a") as f:
            f.write(json.dumps({"test": os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0],
                                "what": what, "n": int(np.asarray(ref).size),
                                "max_rel": mr, "normwise": nw, "element": el}) + "\n")
    assert np.all(np.isfinite(np.asarray(got, dtype=np.float64))), f"{what}: non-finite output"
    assert mr <= MAX_REL and nw <= NORMWISE and el <= ELEMENT, \
        f"{what}: max_rel={mr:.3e} normwise={nw:.3e} element={el:.3e}"
    return mr, nw


def assert_gates(got, ref):
    np.testing.assert_allclose(np.asarray(got, np.float64), np.asarray(ref, np.float64),
                               rtol=GATE_RTOL, atol=GATE_ATOL)


def host(t):
    return t.detach().cpu().numpy()


def bits(t):
    return workloads.bf16_bits(t)


def oracle_route(w, logits, sel_bias):
    z = host(logits)
    if w.score_fn == "softmax":
        return oracle.route_softmax(z, w.k)
    b = None if sel_bias is None else host(sel_bias)
    return oracle.route_sigmoid_group(z, b, w.k, w.n_group, w.topk_group, w.route_scale)


def oracle_capacity(w):
    if w.capacity_factor is None:
        return -1
    return oracle.capacity(w.capacity_factor, w.T, w.k, w.E)


def oracle_token_outputs(w, tokens, x_bits, ids, gates, perm, weights_of, shared=None,
                         shared_x_bits=None):
    """Oracle combined output rows for `tokens` (float64 [n, d]) and their y rows by row.

    Each sampled route's expert output is computed from the token row and that
    expert's weights; ``weights_of(e)`` returns expert e's (Wg, Wu, Wd) bf16 bits.
    The shared expert reads ``shared_x_bits`` (default: the routed experts' rows)."""
    if shared_x_bits is None:
        shared_x_bits = x_bits
    k = w.k
    need = {}
    for t in tokens:
        for j in range(k):
            r = t * k + j
            if perm["route_to_row"][r] >= 0:
                need.setdefault(int(ids[t, j]), []).append(r)
    y_of_row = {}
    for e, routes in need.items():
        xr = oracle.bf16_to_f64(x_bits[np.array(routes) // k])
        wg_e, wu_e, wd_e = weights_of(e)
        _, y = oracle.swiglu(xr, oracle.bf16_to_f64(wg_e), oracle.bf16_to_f64(wu_e),
                             oracle.bf16_to_f64(wd_e))
        for i, r in enumerate(routes):
            y_of_row[int(perm["route_to_row"][r])] = y[i]
    sh = None
    if shared is not None:
        sg, su, sd = shared
        _, sh = oracle.swiglu(oracle.bf16_to_f64(shared_x_bits[np.array(tokens)]),
                              oracle.bf16_to_f64(sg[0]), oracle.bf16_to_f64(su[0]),
                              oracle.bf16_to_f64(sd[0]))
    outs = []
    for i, t in enumerate(tokens):
        rows = perm["route_to_row"][t * k:(t + 1) * k]
        acc = oracle.combine_token(lambda r: y_of_row[r], rows, gates[t],
                                   None if sh is None else sh[i])
        outs.append(np.zeros(x_bits.shape[1]) if acc is None else acc)
    return np.stack(outs), y_of_row


def weights_fetcher(wg, wu, wd):
    """Host bf16 bits of one expert's weights, fetched on demand (weights stay on the GPU)."""
    cache = {}

    def get(e):
        if e not in cache:
            cache[e] = (bits(wg[e]), bits(wu[e]), bits(wd[e]))
        return cache[e]
    return get


# ----------------------------------------------------------------------------
# Rows that reach every tile of a grouped GEMM
# ----------------------------------------------------------------------------

TILE_ROWS = 128  # rows of one CTA's tile; a CTA pair's 256-row tile is two of them


def stratified_rows(begins, counts, rng, tile=TILE_ROWS):
    """The first and last row of every non-empty segment and one row drawn from every
    `tile`-row block counted from the segment's start, so the checked rows reach every
    m-tile of every segment (both CTAs of a pair tile, and each segment's ragged last
    block)."""
    rows = set()
    for b, c in zip(np.asarray(begins).tolist(), np.asarray(counts).tolist()):
        if c <= 0:
            continue
        rows.update((b, b + c - 1))
        for t0 in range(0, c, tile):
            rows.add(b + t0 + int(rng.integers(0, min(tile, c - t0))))
    return np.array(sorted(rows), dtype=np.int64)


def assert_every_tile_reached(rows, begins, counts, tile=TILE_ROWS):
    begins = np.asarray(begins, dtype=np.int64)
    counts = np.asarray(counts, dtype=np.int64)
    want = {(q, t) for q, c in enumerate(counts.tolist()) for t in range((c + tile - 1) // tile)}
    q = np.searchsorted(begins, rows, side="right") - 1
    assert np.all(q >= 0) and np.all(rows < begins[q] + counts[q]), "row outside its segment"
    got = set(zip(q.tolist(), ((rows - begins[q]) // tile).tolist()))
    assert got == want, f"{len(want - got)} of {len(want)} (segment, m-tile) pairs not reached"


def oracle_expert_rows(rows, expert_of_row, x_rows_bits, weights_of, threads=16):
    """Oracle (h, y) float64 for each row in `rows`: expert ``expert_of_row[i]``'s SwiGLU
    of the bf16 row ``x_rows_bits[i]``.  Rows are grouped by expert so each expert's
    weights are converted once; experts run on a thread pool (numpy releases the
    interpreter lock in its conversions and products)."""
    from concurrent.futures import ThreadPoolExecutor
    rows = np.asarray(rows)
    expert_of_row = np.asarray(expert_of_row)
    groups = {}
    for i, e in enumerate(expert_of_row.tolist()):
        groups.setdefault(e, []).append(i)

    def one(item):
        e, idx = item
        wg_e, wu_e, wd_e = weights_of(e)
        h, y = oracle.swiglu(oracle.bf16_to_f64(x_rows_bits[idx]), oracle.bf16_to_f64(wg_e),
                             oracle.bf16_to_f64(wu_e), oracle.bf16_to_f64(wd_e))
        return idx, h, y

    h_all = y_all = None
    with ThreadPoolExecutor(max_workers=threads) as ex:
        for idx, h, y in ex.map(one, groups.items()):
            if h_all is None:
                h_all = np.zeros((rows.size, h.shape[1]))
                y_all = np.zeros((rows.size, y.shape[1]))
            h_all[idx] = h
            y_all[idx] = y
    return h_all, y_all


def weights_fetcher_uncached(wg, wu, wd):
    """Host bf16 bits of one expert's weights, fetched on every call (for walks over many
    experts whose weights would not all fit a host cache comfortably)."""
    return lambda e: (bits(wg[e]), bits(wu[e]), bits(wd[e]))
