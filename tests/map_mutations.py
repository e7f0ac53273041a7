"""One-field (and order-only) mutations of the dispatch maps, for the negative tests
of the map validators and of the oracle's invariant checks.

Each generator takes a valid set of maps as plain integer arrays and yields
``(name, maps)`` pairs in which one entry was changed (or two rows were swapped
consistently in both directions of a map, which keeps the bijection and breaks
only the order).  Every yielded case breaks at least one invariant by
construction; the comment at each case says which.  Index manipulation only:
nothing here computes a route, a count or a payload.
"""
import numpy as np


def _copy(maps):
    return {k: (np.array(v, copy=True) if isinstance(v, np.ndarray) else v)
            for k, v in maps.items()}


def permutation_mutations(maps, E, cap, live_routes):
    """maps: counts [E], offsets [E+1], row_to_route [>= offsets[E]], route_to_row [R],
    n_dropped (int).  Routes at or past live_routes are padding."""
    counts, offsets = maps["counts"], maps["offsets"]
    r2r, row2 = maps["route_to_row"], maps["row_to_route"]
    acc = int(offsets[E])
    R = r2r.size
    full = [e for e in range(E) if counts[e] >= 2]
    out = []

    m = _copy(maps); m["counts"][int(np.argmax(counts))] += 1; out.append(("count+1", m))
    m = _copy(maps); m["offsets"][E] -= 1; out.append(("sentinel-1", m))
    m = _copy(maps); m["offsets"][0] = 1; out.append(("offsets[0]=1", m))
    m = _copy(maps); m["n_dropped"] = maps["n_dropped"] + 1; out.append(("n_dropped+1", m))
    if E > 1:
        e = max(range(1, E), key=lambda x: counts[x - 1])
        m = _copy(maps); m["offsets"][e] += 1; out.append(("inner-offset+1", m))
    if acc >= 2:
        # a row points at another accepted route (which does not point back)
        m = _copy(maps); m["row_to_route"][0] = row2[1]; out.append(("row_to_route[0]", m))
        # a route points at another route's row
        r = int(row2[0])
        m = _copy(maps); m["route_to_row"][r] = 1; out.append(("route_to_row[r]", m))
        # an accepted route marked dropped (its row keeps pointing at it)
        m = _copy(maps); m["route_to_row"][r] = -1; out.append(("accepted->dropped", m))
        # an out-of-range row
        m = _copy(maps); m["route_to_row"][r] = acc + 5; out.append(("row out of range", m))
        # a row that names a route id outside the live routes
        m = _copy(maps); m["row_to_route"][acc - 1] = R + 3; out.append(("route out of range", m))
    if full:
        # swap two rows of one segment in both maps: bijection kept, order broken
        e = full[0]
        i = int(offsets[e])
        m = _copy(maps)
        a, b = int(row2[i]), int(row2[i + 1])
        m["row_to_route"][i], m["row_to_route"][i + 1] = b, a
        m["route_to_row"][a], m["route_to_row"][b] = i + 1, i
        out.append(("stable-order swap", m))
    nz = [e for e in range(E) if counts[e] >= 1]
    if len(nz) >= 2:
        # swap the first rows of two segments in both maps: routes in foreign segments
        i, j = int(offsets[nz[0]]), int(offsets[nz[1]])
        m = _copy(maps)
        a, b = int(row2[i]), int(row2[j])
        m["row_to_route"][i], m["row_to_route"][j] = b, a
        m["route_to_row"][a], m["route_to_row"][b] = j, i
        out.append(("cross-segment swap", m))
    dropped = [r for r in range(min(R, live_routes)) if r2r[r] == -1]
    if dropped and acc >= 1:
        # a dropped route given an accepted row
        m = _copy(maps); m["route_to_row"][dropped[0]] = 0; out.append(("dropped->row", m))
    if cap >= 0 and dropped:
        # admission order: a dropped route takes the row of an earlier accepted
        # route of its expert, which becomes the dropped one (counts unchanged)
        ids = maps["ids"]
        for rd in dropped:
            e = int(ids[rd])
            if 0 <= e < E and counts[e] >= 1:
                i = int(offsets[e])
                ra = int(row2[i])
                m = _copy(maps)
                m["row_to_route"][i] = rd
                m["route_to_row"][rd], m["route_to_row"][ra] = i, -1
                out.append(("admission order", m))
                break
    if live_routes < R:
        m = _copy(maps); m["route_to_row"][R - 1] = 0; out.append(("padding mapped", m))
    return out


def pool_mutations(maps, n_dest, L, pool_cap):
    """maps: headers [n_dest, d] (pool row 0), route_to_poolrow [R], fill [n_dest]."""
    hdr, where, fill = maps["headers"], maps["route_to_poolrow"], maps["fill"]
    placed = [r for r in range(where.size) if where[r] >= 0]
    out = []
    D = int(np.argmax(fill))
    if fill[D] >= 1:
        m = _copy(maps)
        m["headers"][D, 0] = (hdr[D, 0] + 1) % L if L > 1 else 0xFFFF
        out.append(("header id", m))
        m = _copy(maps); m["fill"][D] -= 1; out.append(("fill-1", m))
    if fill[D] < pool_cap:
        m = _copy(maps); m["headers"][D, fill[D]] = 0; out.append(("header past fill", m))
        m = _copy(maps); m["fill"][D] += 1; out.append(("fill+1", m))
    m = _copy(maps); m["fill"][D] = pool_cap + 1; out.append(("fill>cap", m))
    if len(placed) >= 2:
        m = _copy(maps); m["route_to_poolrow"][placed[0]] = where[placed[1]]
        out.append(("two routes one row", m))
        m = _copy(maps); m["route_to_poolrow"][placed[0]] = -1; out.append(("placed->unplaced", m))
    unplaced = [r for r in range(where.size) if where[r] == -1]
    if unplaced and placed:
        m = _copy(maps); m["route_to_poolrow"][unplaced[0]] = where[placed[0]]
        out.append(("unplaced->row", m))
    # two routes of one pool with the same local id swap rows: order broken only
    by_row = {int(where[r]): r for r in placed}
    for p in sorted(by_row):
        q = p + 1
        if q in by_row and q // pool_cap == p // pool_cap and \
                hdr[p // pool_cap, p % pool_cap] == hdr[q // pool_cap, q % pool_cap]:
            m = _copy(maps)
            m["route_to_poolrow"][by_row[p]], m["route_to_poolrow"][by_row[q]] = q, p
            out.append(("pool order swap", m))
            break
    return out


def compact_mutations(maps, n_local, local_cap):
    """maps: headers [n_src, >= pool_cap], local_counts [n_local], poolrow_to_row [n_src*pool_cap]."""
    cnt, p2r, hdr = maps["local_counts"], maps["poolrow_to_row"], maps["headers"]
    pool_cap = p2r.size // hdr.shape[0]
    mapped = [i for i in range(p2r.size) if p2r[i] >= 0]
    out = []
    l = int(np.argmax(cnt))
    if cnt[l] < local_cap:
        m = _copy(maps); m["local_counts"][l] += 1; out.append(("count+1", m))
    if cnt[l] >= 1:
        m = _copy(maps); m["local_counts"][l] -= 1; out.append(("count-1", m))
    m = _copy(maps); m["local_counts"][l] = local_cap + 1; out.append(("count>cap", m))
    if len(mapped) >= 2:
        m = _copy(maps); m["poolrow_to_row"][mapped[0]] = p2r[mapped[1]]
        out.append(("two rows one slot", m))
    if mapped:
        m = _copy(maps); m["poolrow_to_row"][mapped[0]] = -1; out.append(("mapped->-1", m))
        i = mapped[0]
        s, r = divmod(i, pool_cap)
        m = _copy(maps)
        m["headers"][s, r] = (hdr[s, r] + 1) % n_local if n_local > 1 else 0xFFFF
        out.append(("header of mapped row", m))
    by_slot = {int(p2r[i]): i for i in mapped}
    for q in sorted(by_slot):
        if q + 1 in by_slot and (q + 1) // local_cap == q // local_cap:
            m = _copy(maps)
            m["poolrow_to_row"][by_slot[q]], m["poolrow_to_row"][by_slot[q + 1]] = q + 1, q
            out.append(("slot order swap", m))
            break
    return out
