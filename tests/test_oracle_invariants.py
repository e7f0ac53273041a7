"""The oracle's map invariant checks and expert demand, pinned: they accept the maps
the pages print (M6.2 Loop 9) and maps built by brute force in this file, and
they reject every one-field mutation of those maps ([M6.6] 0x0CD "Route And
Combine Assertions"; the pages' own fixtures reject one-field mutations the same
way).  CPU only."""
import json
import os

import numpy as np
import pytest

import oracle
from map_mutations import compact_mutations, permutation_mutations, pool_mutations

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _brute_permute(flat, E, cap, live):
    """Admission in route id order, rows by (expert, route id): written as loops."""
    seen, acc = [0] * E, []
    for r in range(live):
        e = flat[r]
        if cap < 0 or seen[e] < cap:
            acc.append(r)
        seen[e] += 1
    rows = sorted(acc, key=lambda r: (flat[r], r))
    counts = [sum(1 for r in acc if flat[r] == e) for e in range(E)]
    offsets = [0]
    for c in counts:
        offsets.append(offsets[-1] + c)
    r2r = [-1] * len(flat)
    for i, r in enumerate(rows):
        r2r[r] = i
    return dict(ids=np.array(flat), counts=np.array(counts), offsets=np.array(offsets),
                row_to_route=np.array(rows + [0] * (len(flat) - len(rows)), dtype=np.int64),
                route_to_row=np.array(r2r), n_dropped=live - len(acc))


def _random_case(rng, with_padding):
    T, E = int(rng.integers(1, 9)), int(rng.integers(1, 7))
    k = int(rng.integers(1, min(E, 3) + 1))
    flat = [int(v) for v in np.concatenate([rng.permutation(E)[:k] for _ in range(T)])]
    live = T * k
    if with_padding and T > 1:
        live = int(rng.integers(0, T)) * k
        flat = flat[:live] + [-1] * (T * k - live)
    cap = int(rng.choice([-1, 0, 1, 2, 3]))
    return flat, E, cap, live


def _check(maps, E, cap, live):
    return oracle.permutation_violations(maps["ids"], E, cap, maps["counts"], maps["offsets"],
                                         maps["row_to_route"], maps["route_to_row"],
                                         maps["n_dropped"], live)


def test_checks_accept_the_page_fixture():
    with open(os.path.join(GOLDEN, "m62_loop9_permute_combine.json")) as f:
        fx = json.load(f)
    ids = np.array(fx["expert_of_route"])
    assert oracle.permutation_violations(ids, fx["E"], -1, fx["counts"], fx["offsets"], fx["pi"],
                                         fx["inverse_pi"], 0) == []
    # dropless: the demand is the admitted count the page prints
    assert oracle.expert_demand(ids, fx["E"]).tolist() == fx["counts"]


@pytest.mark.parametrize("padding", [False, True])
def test_checks_accept_brute_force_and_oracle_permutations(padding):
    rng = np.random.default_rng(21 + padding)
    for _ in range(150):
        flat, E, cap, live = _random_case(rng, padding)
        bf = _brute_permute(flat, E, cap, live)
        assert _check(bf, E, cap, live) == []
        if not padding:
            p = oracle.permute(np.array(flat), E, cap)
            assert oracle.permutation_violations(flat, E, cap, p["counts"], p["offsets"],
                                                 p["row_to_route"], p["route_to_row"],
                                                 p["n_dropped"]) == []


@pytest.mark.parametrize("padding", [False, True])
def test_every_permutation_mutation_is_flagged(padding):
    rng = np.random.default_rng(31 + padding)
    seen = set()
    for _ in range(150):
        flat, E, cap, live = _random_case(rng, padding)
        bf = _brute_permute(flat, E, cap, live)
        for name, m in permutation_mutations(bf, E, cap, live):
            assert _check(m, E, cap, live) != [], (name, flat, E, cap, live)
            seen.add(name)
    # the families the mutation set is meant to cover all occurred
    must = {"count+1", "sentinel-1", "n_dropped+1", "row_to_route[0]", "route_to_row[r]",
            "accepted->dropped", "stable-order swap", "cross-segment swap", "dropped->row",
            "admission order"}
    if padding:
        must.add("padding mapped")
    assert must <= seen, must - seen


def test_expert_demand_brute_force_and_capacity_law():
    rng = np.random.default_rng(41)
    for _ in range(100):
        flat, E, cap, live = _random_case(rng, True)
        n = oracle.expert_demand(flat, E, live)
        assert n.tolist() == [sum(1 for r in range(live) if flat[r] == e) for e in range(E)]
        bf = _brute_permute(flat, E, cap, live)
        # admitted count = min(n_e, C); dropless admits everything
        assert bf["counts"].tolist() == [min(v, cap) if cap >= 0 else v for v in n.tolist()]


# ----------------------------------------------------------------------------
# Pooled layout
# ----------------------------------------------------------------------------

def _brute_pack(flat, n_dest, L, n_waves, cap, wave, policy, d):
    seen = [0] * n_dest
    fill = [0] * n_dest
    hdr = np.full((n_dest, d), 0xFFFF, dtype=np.int64)
    where = np.full(len(flat), -1, dtype=np.int64)
    for r, e in enumerate(flat):
        D, l = e // L, e % L
        j = seen[D]
        seen[D] += 1
        w, row = (j % n_waves, j // n_waves) if policy == "stripe" else (D % n_waves, j)
        if w == wave and row < cap:
            hdr[D, row] = l
            where[r] = D * cap + row
            fill[D] += 1
    return dict(headers=hdr, route_to_poolrow=where, fill=np.array(fill))


def _brute_compact(hdr, cap, n_local, local_cap):
    cnt = [0] * n_local
    out = np.full(hdr.shape[0] * cap, -1, dtype=np.int64)
    for s in range(hdr.shape[0]):
        for r in range(cap):
            l = int(hdr[s, r])
            if l >= n_local:
                continue
            if cnt[l] < local_cap:
                out[s * cap + r] = l * local_cap + cnt[l]
            cnt[l] += 1
    return dict(headers=hdr.copy(), local_counts=np.array([min(c, local_cap) for c in cnt]),
                poolrow_to_row=out)


@pytest.mark.parametrize("policy", ["stripe", "destmod"])
def test_pool_checks_accept_valid_and_flag_mutations(policy):
    rng = np.random.default_rng(51)
    seen_p, seen_c = set(), set()
    for _ in range(80):
        n_dest, L, n_waves = int(rng.integers(1, 5)), int(rng.integers(1, 4)), int(rng.integers(1, 4))
        E = n_dest * L
        T = int(rng.integers(1, 12))
        k = int(rng.integers(1, min(E, 3) + 1))
        flat = [int(v) for v in np.concatenate([rng.permutation(E)[:k] for _ in range(T)])]
        cap = int(rng.integers(1, 5))
        d = cap + int(rng.integers(0, 3))
        lcap = int(rng.integers(1, 6))
        for wave in range(n_waves):
            pk = _brute_pack(flat, n_dest, L, n_waves, cap, wave, policy, d)
            assert oracle.pool_violations(flat, n_dest, L, cap, pk["headers"],
                                          pk["route_to_poolrow"], pk["fill"]) == []
            for name, m in pool_mutations(pk, n_dest, L, cap):
                assert oracle.pool_violations(flat, n_dest, L, cap, m["headers"],
                                              m["route_to_poolrow"], m["fill"]) != [], name
                seen_p.add(name)
            cp = _brute_compact(pk["headers"], cap, L, lcap)
            assert oracle.compact_violations(cp["headers"], cap, L, lcap, cp["local_counts"],
                                             cp["poolrow_to_row"]) == []
            for name, m in compact_mutations(cp, L, lcap):
                assert oracle.compact_violations(m["headers"], cap, L, lcap, m["local_counts"],
                                                 m["poolrow_to_row"]) != [], name
                seen_c.add(name)
    assert {"header id", "fill-1", "fill+1", "two routes one row", "placed->unplaced",
            "pool order swap"} <= seen_p
    assert {"count+1", "count-1", "two rows one slot", "mapped->-1", "header of mapped row",
            "slot order swap"} <= seen_c


def test_compact_checks_follow_the_receiver_rotation():
    rng = np.random.default_rng(71)
    n_dest, L, cap, lcap = 5, 2, 6, 4
    pools = np.zeros((n_dest, cap + 1, 8), np.uint16)
    pools[:, 0, :] = oracle.EMPTY_HEADER
    for D in range(n_dest):
        f = int(rng.integers(2, cap + 1))
        pools[D, 0, :f] = rng.integers(0, L, f)
    hdr = pools[:, 0, :]
    for first in range(n_dest):
        cp = oracle.pool_compact(pools, cap, L, lcap, first)
        assert oracle.compact_violations(hdr, cap, L, lcap, cp["local_counts"],
                                         cp["poolrow_to_row"], first) == []
        if first:
            # the same maps read with the fixed source order break the order checks
            assert oracle.compact_violations(hdr, cap, L, lcap, cp["local_counts"],
                                             cp["poolrow_to_row"], 0) != []


def test_pool_checks_accept_the_oracle_layout():
    rng = np.random.default_rng(61)
    n_dest, L, n_waves, cap, lcap, T, k, d = 4, 3, 3, 5, 6, 40, 3, 8
    ids = np.stack([rng.permutation(n_dest * L)[:k] for _ in range(T)])
    x = rng.integers(0, 2**15, size=(T, d)).astype(np.uint16)
    for policy in ("stripe", "destmod"):
        for wave in range(n_waves):
            pk = oracle.pool_pack(ids, x, n_dest, L, n_waves, cap, wave, policy)
            assert oracle.pool_violations(ids, n_dest, L, cap, pk["pools"][:, 0, :],
                                          pk["route_to_poolrow"], pk["fill"]) == []
            cp = oracle.pool_compact(pk["pools"], cap, L, lcap)
            assert oracle.compact_violations(pk["pools"][:, 0, :], cap, L, lcap,
                                             cp["local_counts"], cp["poolrow_to_row"]) == []
