"""Device map validators, expert demand and the bounded-wait self-test, through the
C ABI.  The validators ([M6.6] 0x0CD "Route And Combine Assertions") must pass
on the maps the permute and pool kernels write, and flag every one-field
mutation of those maps; the oracle's invariant checks must reach the same
verdict on the same host copies, case by case."""
import numpy as np
import pytest
import torch

import oracle
from map_mutations import compact_mutations, permutation_mutations, pool_mutations
from moe_check import host

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


def i32(a):
    return torch.from_numpy(np.ascontiguousarray(np.asarray(a), dtype=np.int32)).to(DEV)


def status0():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def _skewed_ids(rng, T, E, k, alpha=0.5):
    p = rng.dirichlet(np.ones(E) * alpha)
    return np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)


# ----------------------------------------------------------------------------
# Permutation
# ----------------------------------------------------------------------------

def _permute(T, d, E, k, cap, ids_np, valid=None):
    """Run moe_permute (or the bucket variant when valid is given); host copies of the maps."""
    g = G()
    R = T * k
    ids = i32(ids_np)
    x = torch.zeros((T, d), dtype=torch.bfloat16, device=DEV)
    xp = torch.empty((max(R, 1), d), dtype=torch.bfloat16, device=DEV)
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    r2r = torch.zeros(max(R, 1), dtype=torch.int32, device=DEV)
    inv = torch.empty(max(R, 1), dtype=torch.int32, device=DEV)
    nd = torch.zeros(1, dtype=torch.int32, device=DEV)
    wsb = g.moe_permute_workspace_size(T, k, E)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    st = status0()
    if valid is None:
        g.moe_permute(T, d, E, k, cap, ids, x, xp, counts, offsets, r2r, inv, nd, ws, wsb, st)
    else:
        g.moe_permute_bucket(T, d, E, k, cap, i32([valid]), ids, x, xp, counts, offsets, r2r, inv,
                             nd, ws, wsb, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return dict(ids=np.asarray(ids_np).reshape(-1).astype(np.int64), counts=host(counts),
                offsets=host(offsets), row_to_route=host(r2r)[:R], route_to_row=host(inv)[:R],
                n_dropped=int(nd.item()))


def _validate_perm(T, E, k, cap, valid, m):
    g = G()
    st = status0()
    g.moe_validate_permutation(T, E, k, cap, None if valid is None else i32([valid]), i32(m["ids"]),
                               i32(m["counts"]), i32(m["offsets"]),
                               i32(m["row_to_route"] if m["row_to_route"].size else [0]),
                               i32(m["route_to_row"] if m["route_to_row"].size else [0]),
                               i32([m["n_dropped"]]), st)
    torch.cuda.synchronize()
    return int(st.item())


@pytest.mark.parametrize("T,d,E,k,cap,valid", [
    (256, 64, 8, 2, 80, None),        # capacity with drops
    (300, 64, 128, 8, -1, None),      # dropless, many experts
    (5000, 64, 32, 4, 600, None),     # several permute tiles, drops
    (4096, 64, 8, 2, 0, None),        # capacity 0: everything dropped
    (1, 64, 4, 4, -1, None),          # one token, k = E
    (300, 64, 32, 4, 100, 211),       # token bucket: padding slots
    (300, 64, 32, 4, -1, 0),          # token bucket with no real token
])
def test_permutation_validator_passes_and_flags_mutations(T, d, E, k, cap, valid):
    g = G()
    rng = np.random.default_rng(T + E + k)
    ids_np = _skewed_ids(rng, T, E, k)
    if valid is not None:
        ids_np[valid:] = g.MOE_ROUTE_MASKED
    m0 = _permute(T, d, E, k, cap, ids_np, valid)
    live = T * k if valid is None else valid * k
    assert oracle.permutation_violations(m0["ids"], E, cap, m0["counts"], m0["offsets"],
                                         m0["row_to_route"], m0["route_to_row"], m0["n_dropped"],
                                         live) == []
    assert _validate_perm(T, E, k, cap, valid, m0) == 0
    muts = permutation_mutations(m0, E, cap, live)
    assert muts
    for name, m in muts:
        ora = oracle.permutation_violations(m["ids"], E, cap, m["counts"], m["offsets"],
                                            m["row_to_route"], m["route_to_row"], m["n_dropped"],
                                            live)
        st = _validate_perm(T, E, k, cap, valid, m)
        assert ora != [], name
        assert st & g.MOE_DEV_BAD_MAP, (name, ora)


@pytest.mark.parametrize("T,E,k,cap", [(8192, 256, 8, 256), (4096, 8, 2, -1)])
def test_permutation_validator_at_full_size(T, E, k, cap):
    """The V3 (capacity 256) and prefill (dropless) routing sizes: passes on the real
    maps, flags an order swap deep inside the route range."""
    g = G()
    rng = np.random.default_rng(E)
    ids_np = _skewed_ids(rng, T, E, k, alpha=2.0)
    m0 = _permute(T, 64, E, k, cap, ids_np)
    assert _validate_perm(T, E, k, cap, None, m0) == 0
    names = {n: m for n, m in permutation_mutations(m0, E, cap, T * k)}
    for n in ("stable-order swap", "cross-segment swap", "n_dropped+1", "route_to_row[r]"):
        assert _validate_perm(T, E, k, cap, None, names[n]) & g.MOE_DEV_BAD_MAP, n


# ----------------------------------------------------------------------------
# Pooled layout
# ----------------------------------------------------------------------------

def _hdr_host(pools):
    return host(pools.view(torch.int16)[:, 0, :]).astype(np.int64) & 0xFFFF


def _pools_with_headers(pools, headers):
    out = pools.clone()
    out.view(torch.int16)[:, 0, :] = torch.from_numpy(
        headers.astype(np.uint16).view(np.int16)).to(DEV)
    return out


@pytest.mark.parametrize("policy", [0, 1])
@pytest.mark.parametrize("T,d,k,n_dest,L,n_waves,pool_cap,local_cap", [
    (600, 64, 4, 8, 3, 3, 40, 50),    # sender and receiver drops
    (200, 128, 2, 4, 2, 2, 128, 400), # no drops, header as wide as the row
    (1, 64, 1, 2, 1, 1, 4, 4),
])
def test_pool_validators_pass_and_flag_mutations(policy, T, d, k, n_dest, L, n_waves, pool_cap,
                                                 local_cap):
    g = G()
    rng = np.random.default_rng(T + d)
    E = n_dest * L
    ids_np = _skewed_ids(rng, T, E, k)
    ids = i32(ids_np)
    x = torch.randn((T, d), device=DEV).to(torch.bfloat16)
    pp = g.PoolParams(n_dest, L, n_waves, pool_cap, policy)
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
    vpb = g.moe_validate_pools_workspace_size(pp)
    vp = torch.empty(vpb, dtype=torch.uint8, device=DEV)
    vcb = g.moe_validate_compact_workspace_size(L, local_cap)
    vc = torch.empty(vcb, dtype=torch.uint8, device=DEV)

    def check_pack(m, pools_t):
        st = status0()
        g.moe_validate_pools(pp, T, d, k, ids, pools_t, i32(m["route_to_poolrow"]), i32(m["fill"]),
                             vp, vpb, st)
        torch.cuda.synchronize()
        return int(st.item())

    def check_compact(m, pools_t):
        st = status0()
        g.moe_validate_compact(n_dest, pool_cap, d, L, local_cap, pools_t, i32(m["local_counts"]),
                               i32(m["poolrow_to_row"]), vc, vcb, st)
        torch.cuda.synchronize()
        return int(st.item())

    for wave in range(n_waves):
        st = status0()
        g.moe_pool_pack(pp, T, d, k, wave, ids, x, pools, r2p, fill, sdrop, pws, pwsb, st)
        g.moe_pool_compact(n_dest, pool_cap, d, L, local_cap, pools, compact, lcounts, p2r, rdrop,
                           cws, cwsb, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        hdr = _hdr_host(pools)
        pk = dict(headers=hdr, route_to_poolrow=host(r2p).astype(np.int64),
                  fill=host(fill).astype(np.int64))
        assert oracle.pool_violations(ids_np, n_dest, L, pool_cap, hdr, pk["route_to_poolrow"],
                                      pk["fill"]) == []
        assert check_pack(pk, pools) == 0
        for name, m in pool_mutations(pk, n_dest, L, pool_cap):
            assert oracle.pool_violations(ids_np, n_dest, L, pool_cap, m["headers"],
                                          m["route_to_poolrow"], m["fill"]) != [], name
            pm = pools if np.array_equal(m["headers"], hdr) else \
                _pools_with_headers(pools, m["headers"])
            assert check_pack(m, pm) & g.MOE_DEV_BAD_MAP, name
        cp = dict(headers=hdr.copy(), local_counts=host(lcounts).astype(np.int64),
                  poolrow_to_row=host(p2r).astype(np.int64))
        assert oracle.compact_violations(hdr, pool_cap, L, local_cap, cp["local_counts"],
                                         cp["poolrow_to_row"]) == []
        assert check_compact(cp, pools) == 0
        for name, m in compact_mutations(cp, L, local_cap):
            assert oracle.compact_violations(m["headers"], pool_cap, L, local_cap,
                                             m["local_counts"], m["poolrow_to_row"]) != [], name
            pm = pools if np.array_equal(m["headers"], hdr) else \
                _pools_with_headers(pools, m["headers"])
            assert check_compact(m, pm) & g.MOE_DEV_BAD_MAP, name


# ----------------------------------------------------------------------------
# Expert demand
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("T,E,k,valid", [(8192, 256, 8, None), (1, 8, 2, None),
                                         (65536, 384, 8, None), (300, 512, 16, None),
                                         (128, 128, 8, 37), (128, 128, 8, 0)])
def test_expert_demand_parity(T, E, k, valid):
    g = G()
    rng = np.random.default_rng(T + E)
    ids_np = _skewed_ids(rng, T, E, k)
    live = T * k if valid is None else valid * k
    if valid is not None:
        ids_np[valid:] = g.MOE_ROUTE_MASKED
    dem = torch.full((E,), 77, dtype=torch.int32, device=DEV)  # overwritten, not accumulated
    st = status0()
    g.moe_expert_demand(T, k, E, None if valid is None else i32([valid]), i32(ids_np), dem, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert host(dem).tolist() == oracle.expert_demand(ids_np, E, live).tolist()


def test_expert_demand_reports_bad_ids_and_skips_masked():
    g = G()
    ids_np = np.array([[0, 1], [2, 99], [3, -1]], np.int32)
    dem = torch.empty(4, dtype=torch.int32, device=DEV)
    st = status0()
    g.moe_expert_demand(3, 2, 4, None, i32(ids_np), dem, st)
    torch.cuda.synchronize()
    assert int(st.item()) & g.MOE_DEV_BAD_EXPERT_ID
    assert host(dem).tolist() == [1, 1, 1, 1]
    st = status0()
    g.moe_expert_demand(3, 2, 4, None, i32(np.where(ids_np == 99, 1, ids_np)), dem, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0  # MOE_ROUTE_MASKED is not an error
    assert host(dem).tolist() == [1, 2, 1, 1]


# ----------------------------------------------------------------------------
# Bounded wait
# ----------------------------------------------------------------------------

def test_bounded_wait_gives_up_with_timeout_status_and_context_survives():
    """A wait on a barrier nothing arrives at gives up after its limit: the status
    word says MOE_DEV_TIMEOUT, and the context keeps working afterwards."""
    g = G()
    st = status0()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    g.moe_debug_wait_timeout(2_000_000, st)  # 2 ms
    stop.record()
    torch.cuda.synchronize()
    assert int(st.item()) == g.MOE_DEV_TIMEOUT
    assert 1.5 <= start.elapsed_time(stop) < 1000.0
    rng = np.random.default_rng(0)
    m = _permute(64, 64, 8, 2, -1, _skewed_ids(rng, 64, 8, 2))
    assert _validate_perm(64, 8, 2, -1, None, m) == 0


def test_compact_validator_follows_the_rotation():
    """The compact validator checks slots in the receiver's visiting order: it passes the
    rotated compact's maps with the same first source and flags them read in fixed
    source order, as the oracle's checks do."""
    g = G()
    rng = np.random.default_rng(5)
    n_src, pool_cap, d, L, local_cap = 6, 16, 64, 2, 12
    pools = torch.zeros((n_src, pool_cap + 1, d), dtype=torch.bfloat16, device=DEV)
    hdr = np.full((n_src, d), 0xFFFF, np.int64)
    for s_ in range(n_src):
        f = int(rng.integers(4, pool_cap + 1))
        hdr[s_, :f] = rng.integers(0, L, f)
    pools.view(torch.int16)[:, 0, :] = torch.from_numpy(hdr.astype(np.uint16).view(np.int16)).to(DEV)
    i32 = dict(dtype=torch.int32, device=DEV)
    compact = torch.zeros((L * local_cap, d), dtype=torch.bfloat16, device=DEV)
    lcounts, p2r, rdrop = torch.empty(L, **i32), torch.empty(n_src * pool_cap, **i32), torch.zeros(1, **i32)
    cwsb = g.moe_pool_compact_workspace_size(n_src, pool_cap, L)
    cws = torch.empty(cwsb, dtype=torch.uint8, device=DEV)
    vcb = g.moe_validate_compact_workspace_size(L, local_cap)
    vc = torch.empty(vcb, dtype=torch.uint8, device=DEV)
    first = 3
    st = status0()
    g.moe_pool_compact_rotated(n_src, pool_cap, d, L, local_cap, first, pools, compact, lcounts,
                               p2r, rdrop, cws, cwsb, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for f_check in (first, 0):
        ora = oracle.compact_violations(hdr, pool_cap, L, local_cap, host(lcounts), host(p2r),
                                        f_check)
        st = status0()
        g.moe_validate_compact(n_src, pool_cap, d, L, local_cap, pools, lcounts, p2r, vc, vcb,
                               st, first_source=f_check)
        torch.cuda.synchronize()
        assert (ora == []) == (int(st.item()) == 0), (f_check, ora)
        assert (ora == []) == (f_check == first)
