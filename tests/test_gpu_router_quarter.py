"""The quarter-row router against the warp-per-token router and the oracle.

moe_route selects with four lanes per token for softmax batches of tens of
thousands of tokens (E = 128, 256, 384 or 512, k <= 16) and with one warp per
token otherwise.  Routing the same logits once whole and once in slices of 2,048
tokens runs both kernels on every row: ids and gates must agree bit for bit, the
NaN report must agree, and a sample of rows must match the oracle ([M6.2] 0x06L1:
softmax over the selected top-k, ties to the lower expert).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from moe_check import assert_gates, host

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
T_BIG = 40960 + 7  # above the four-lane kernel's threshold on 152 SMs; a ragged last batch
SLICE = 2048


@pytest.fixture(scope="module", autouse=True)
def built():
    from grouped_expert_gemm_gb300 import build
    build.build()


def g():
    import grouped_expert_gemm_gb300 as m
    return m


def _route(logits, k, valid=None):
    """moe_route (or moe_route_bucket) over all rows in one call."""
    T, E = logits.shape
    p = g().RouteParams(T, E, k, g().MOE_SCORE_SOFTMAX, 0, 0, 1.0)
    ids = torch.full((T, k), -7, dtype=torch.int32, device=DEV)
    gates = torch.full((T, k), -7.0, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    if valid is None:
        g().moe_route(p, logits, None, ids, gates, st)
    else:
        vt = torch.tensor([valid], dtype=torch.int32, device=DEV)
        g().moe_route_bucket(p, vt, logits, None, ids, gates, st)
    torch.cuda.synchronize()
    return ids, gates, int(st.item())


def _route_sliced(logits, k):
    """The same rows routed SLICE at a time (below the four-lane kernel's threshold)."""
    T, E = logits.shape
    ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
    gates = torch.empty((T, k), dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    for s in range(0, T, SLICE):
        n = min(SLICE, T - s)
        p = g().RouteParams(n, E, k, g().MOE_SCORE_SOFTMAX, 0, 0, 1.0)
        g().moe_route(p, logits[s:s + n], None, ids[s:s + n], gates[s:s + n], st)
    torch.cuda.synchronize()
    return ids, gates, int(st.item())


def _same_bits(a, b):
    return torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.parametrize("E,k", [(384, 8), (128, 8), (256, 6), (512, 16), (384, 1), (128, 12)])
def test_quarter_router_equals_the_warp_router(E, k):
    w = workloads.scaled(workloads.pooled(), T=T_BIG, E=E, k=k)
    logits, _ = workloads.make_router_inputs(w, DEV)
    ids, gates, st = _route(logits, k)
    rids, rgates, rst = _route_sliced(logits, k)
    assert st == 0 and rst == 0
    assert torch.equal(ids, rids)
    assert _same_bits(gates, rgates)
    # and a sample of rows (the first ones and the ragged last batch) against the oracle
    rows = np.r_[0:256, T_BIG - 64:T_BIG]
    oids, ogates = oracle.route_softmax(host(logits)[rows], k)
    assert np.array_equal(host(ids)[rows], oids)
    assert_gates(host(gates)[rows], ogates)


def _edge_logits(T, E, seed):
    """Rows of every awkward kind, cycled: heavy ties with signed zeros, all equal,
    +-inf, scattered NaN, all NaN, one dominant value, and plain normals."""
    rng = np.random.default_rng(seed)
    z = rng.standard_normal((T, E)).astype(np.float32)
    kinds = np.arange(T) % 8
    tie = rng.choice(np.array([-1.0, -0.0, 0.0, 0.5, 2.0], np.float32), size=(T, E))
    z[kinds == 0] = tie[kinds == 0]
    z[kinds == 1] = 0.25
    inf_rows = np.flatnonzero(kinds == 2)
    z[inf_rows, rng.integers(0, E, inf_rows.size)] = np.inf
    z[inf_rows, rng.integers(0, E, inf_rows.size)] = -np.inf
    nan_rows = np.flatnonzero(kinds == 3)
    for c in range(5):
        z[nan_rows, rng.integers(0, E, nan_rows.size)] = np.nan
    z[kinds == 4] = np.nan
    big = np.flatnonzero(kinds == 5)
    z[big, rng.integers(0, E, big.size)] = 1e30
    neg = np.flatnonzero(kinds == 6)
    z[neg] = -np.abs(z[neg])  # every score negative, some -0.0
    z[neg, ::7] = -0.0
    return z


@pytest.mark.parametrize("E,k", [(384, 8), (128, 16), (512, 3)])
def test_quarter_router_edge_rows_equal_the_warp_router(E, k):
    z = _edge_logits(T_BIG, E, seed=E + k)
    logits = torch.from_numpy(z).to(DEV)
    ids, gates, st = _route(logits, k)
    rids, rgates, rst = _route_sliced(logits, k)
    assert torch.equal(ids, rids)
    assert _same_bits(gates, rgates)
    assert st == rst
    assert st & g().MOE_DEV_NONFINITE_LOGIT
    # rows without NaN against the oracle (ties to the lower expert, -0 == +0)
    finite = np.flatnonzero(~np.isnan(z).any(axis=1))[:2000]
    fin = finite[np.isfinite(z[finite]).all(axis=1)]
    oids, ogates = oracle.route_softmax(z[fin], k)
    assert np.array_equal(host(ids)[fin], oids)
    assert_gates(host(gates)[fin], ogates)


def test_quarter_router_padding_slots():
    """A bucket whose valid count ends mid-batch: live rows as without padding,
    padding rows masked."""
    E, k, valid = 384, 8, T_BIG - 1000 - 13
    w = workloads.scaled(workloads.pooled(), T=T_BIG, E=E, k=k)
    logits, _ = workloads.make_router_inputs(w, DEV)
    ids, gates, st = _route(logits, k, valid=valid)
    rids, rgates, _ = _route_sliced(logits, k)
    assert st == 0
    assert torch.equal(ids[:valid], rids[:valid])
    assert _same_bits(gates[:valid], rgates[:valid])
    assert bool((ids[valid:] == g().MOE_ROUTE_MASKED).all())
    assert bool((gates[valid:] == 0).all())
