"""Helpers shared by the GPU parity tests: tolerance checks and the oracle's
pipeline on host copies of the inputs the CUDA path received."""
import numpy as np
import torch

import oracle
import workloads

# Floating-point parity bar.  The stated bar pairs a maximum relative error with
# a normwise one; they are read as the relative error in the max norm and in the
# 2-norm:
#   max_rel  = ||x - r||_inf / ||r||_inf   <= 1e-2
#   normwise = ||x - r||_2   / ||r||_2     <= 2e-3
# A secondary element-wise guard, derived from the arithmetic, also holds every
# element: |x_i - r_i| <= 4e-2 * max(|r_i|, rms(r)).  Outputs are bf16 after two
# bf16 roundings (H, then y), each up to 2^-8 relative at the bottom of a binade,
# on top of the tensor cores' own fp32 accumulation; 4e-2 leaves room for a few
# ulps of that and still catches any wrong row, column or operand.
MAX_REL = 1e-2
NORMWISE = 2e-3
ELEMENT = 4e-2
# Gates are fp32 results of a few fp32 operations: relative 2e-6 plus 1e-7 absolute.
GATE_RTOL, GATE_ATOL = 2e-6, 1e-7


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
