"""CPU oracle for the MoE layer hot path (test infrastructure only).

This module is a plain, slow, deliberately unoptimised restatement of what the
hot path computes.  It exists to check the CUDA library and is used only by the
tests, by ``__graft_entry__.smoke()`` and by the benchmark's CPU-baseline leg;
the product path never imports it.  It shares no code with the CUDA path.

Floating point: expert arithmetic is carried in float64 from exact bf16 inputs.
Values are rounded to bf16 (round-to-nearest-even) only where the method stores
a bf16 tensor (the SwiGLU intermediate H and the expert output y); routing
gates and the combined output are produced in float64 and compared to fp32.
Where floating point decides an integer (which experts a token selects), the
oracle takes that decision in fp32, as the router does.

Sources (page title, section):
  [M6.6]  "M6.6 - MoE Runtime Systems: Placement, Dispatch, Kernels, and Topology"
  [M6.2]  "M6.2 - Expert Parallelism and DeepSeek MoE: Load Balancing, Shared
          Experts, and Fine-Grained Routing"
  [POOL]  "Fixed pooled-wave all-to-all for the 8-of-384 MoE"
  [DISP]  "Dispatch and combine: preserve token identity across expert ranks"

Readings where the pages are silent are noted at each function.
"""
from __future__ import annotations

from fractions import Fraction
import math

import numpy as np

EMPTY_HEADER = 0xFFFF  # header element of an empty pool row


# ----------------------------------------------------------------------------
# bf16 helpers (bit-level; no library rounding routine is trusted)
# ----------------------------------------------------------------------------

def bf16_to_f64(bits) -> np.ndarray:
    """uint16 bf16 bits -> float64 (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16(v) -> np.ndarray:
    """float64 -> bf16 bits, one rounding, to nearest with ties to even.

    bf16 keeps 8 significant bits and fp32's exponent range.  For |v| with
    frexp exponent e (v = m * 2^e, 0.5 <= |m| < 1) the bf16 grid spacing is
    2^(e-8) for normal numbers and 2^-133 below 2^-126.  Dividing by a power of
    two is exact, np.rint rounds half to even, and the rounded value is exactly
    representable in fp32, whose top 16 bits are then the bf16 encoding.
    """
    v = np.asarray(v, dtype=np.float64)
    _, e = np.frexp(v)
    q = np.ldexp(1.0, np.maximum(e, -125) - 8)
    r = np.rint(v / q) * q
    with np.errstate(over="ignore"):
        f = r.astype(np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


# ----------------------------------------------------------------------------
# Capacity  ([M6.2] 0x01C "Capacity Converts Dynamic Routing Into Bounded
# Buffers": C = ceil(c_f * T * k / E); [POOL] 04 "Capacity and memory")
# ----------------------------------------------------------------------------

def _ceil_frac(x: Fraction) -> int:
    return -((-x.numerator) // x.denominator)


def capacity(cf: float, T: int, k: int, E: int) -> int:
    """Per-expert capacity ceil(cf * T * k / E), in exact rational arithmetic.

    cf is read as the decimal it is written as (1.25, 1.1, ...), so that a
    product that is an integer on paper is not pushed up by binary rounding.
    """
    return _ceil_frac(Fraction(str(cf)) * T * k / E)


def pool_capacity(cf: float, T: int, k: int, n_dest: int, n_waves: int) -> int:
    """Sender pool rows per destination per wave: ceil(cf * T*k / n_dest / n_waves)."""
    return _ceil_frac(Fraction(str(cf)) * T * k / n_dest / n_waves)


def local_capacity(cf: float, T: int, k: int, n_local: int, n_waves: int) -> int:
    """Receiver rows per local expert per wave: ceil(cf * T*k / n_local / n_waves)."""
    return _ceil_frac(Fraction(str(cf)) * T * k / n_local / n_waves)


# ----------------------------------------------------------------------------
# Routing
# ----------------------------------------------------------------------------

def _order_desc_lowest_index(scores: np.ndarray) -> np.ndarray:
    """Per row, expert indices by (score descending, index ascending).

    A stable sort of the negated scores keeps equal scores in index order;
    +0.0 and -0.0 compare equal and therefore also fall back to index order.
    """
    return np.argsort(-scores, axis=-1, kind="stable")


def route_softmax(logits: np.ndarray, k: int):
    """Top-k over fp32 logits with gates = softmax over the selected logits.

    [M6.2] 0x06L1: the Mixtral family applies an FP32 softmax and renormalises
    the selected top-k probabilities to one, which equals a softmax taken over
    the k selected logits.  Reading: selection is made on the fp32 logits
    themselves (softmax is monotone, and exp can merge distinct logits),
    slot 0 holds the best expert, ties go to the lower expert index.

    Returns ids int32 [T,k] and gates float64 [T,k].
    """
    z = np.asarray(logits, dtype=np.float32)
    ids = _order_desc_lowest_index(z)[:, :k].astype(np.int32)
    zs = np.take_along_axis(z, ids, axis=1).astype(np.float64)
    m = zs.max(axis=1, keepdims=True)
    ez = np.exp(zs - m)
    gates = ez / ez.sum(axis=1, keepdims=True)
    return ids, gates


# Own exp for the sigmoid that decides the grouped router's selection.  The
# selection must come out identical on the CPU and the GPU, so both sides run
# the same fp32 operations in the same order, each one correctly rounded and
# none fused:
#   Cody-Waite range reduction (Cody & Waite, "Software Manual for the
#   Elementary Functions", 1980): n = rint(x*log2(e)), r = (x - n*L1) - n*L2,
#   with L1 = ln2 cut to 16 significant bits (so n*L1 is exact for |n| <= 256)
#   and L2 = ln2 - L1; then e^r by its degree-7 Taylor polynomial in Horner
#   form; then multiplication by 2^n built from the exponent bits.
_LOG2E_F32 = np.float32(1.0 / math.log(2.0))
_LN2_HI_F32 = np.float32(45426.0 / 65536.0)  # round(ln2 * 2^16) / 2^16
_LN2_LO_F32 = np.float32(math.log(2.0) - 45426.0 / 65536.0)
_TAYLOR_F32 = [np.float32(1.0 / math.factorial(i)) for i in range(8)]  # 1/0! .. 1/7!
_EXP_CLAMP_F32 = np.float32(87.0)


def exp_det_f32(x) -> np.ndarray:
    """e^x in fp32 by the fixed recipe above; x is clamped to [-87, 87].

    The clamp keeps 2^n within the normal fp32 range, so no subnormal or
    infinite intermediate appears and both implementations agree exactly.
    """
    x = np.asarray(x, dtype=np.float32)
    x = np.minimum(np.maximum(x, -_EXP_CLAMP_F32), _EXP_CLAMP_F32)
    n = np.rint(x * _LOG2E_F32).astype(np.float32)
    r = (x - n * _LN2_HI_F32) - n * _LN2_LO_F32
    p = _TAYLOR_F32[7]
    for c in _TAYLOR_F32[6::-1]:
        p = p * r + c
    ni = n.astype(np.int32)
    two_n = ((ni + 127).astype(np.uint32) << 23).view(np.float32)
    return (p * two_n).astype(np.float32)


def sigmoid_det_f32(z) -> np.ndarray:
    """sigma(z) = 1 / (1 + e^-z) in fp32 with the fixed exp above."""
    z = np.asarray(z, dtype=np.float32)
    one = np.float32(1.0)
    return (one / (one + exp_det_f32(-z))).astype(np.float32)


def route_sigmoid_group(logits: np.ndarray, sel_bias, k: int, n_group: int, topk_group: int,
                        route_scale: float, return_groups: bool = False):
    """DeepSeek-V3 group-limited routing.

    [M6.2] 0x06A-0x06D and 0x06I: s = sigmoid(z); corrected score
    s~ = s + b (fp32, b is selection-only state); per contiguous logical group
    the score is the sum of its two largest s~; keep the top ``topk_group``
    groups; experts outside them are not eligible; choose the top k experts by
    s~ among the eligible; gate = route_scale * s_e / sum of s over the
    selected experts (the original affinity, not the corrected score).
    Ties resolve to the lower expert index and the lower group index.

    Returns ids int32 [T,k] and gates float64 [T,k] (plus the kept groups
    [T,topk_group] and the group scores [T,n_group] when return_groups).
    """
    z = np.asarray(logits, dtype=np.float32)
    T, E = z.shape
    assert E % n_group == 0
    s = sigmoid_det_f32(z)
    b = np.zeros(E, np.float32) if sel_bias is None else np.asarray(sel_bias, np.float32)
    st = (s + b[None, :]).astype(np.float32)
    grouped = st.reshape(T, n_group, E // n_group)
    top2 = np.take_along_axis(grouped, _order_desc_lowest_index(grouped)[:, :, :2], axis=2)
    gscore = (top2[:, :, 0] + top2[:, :, 1]).astype(np.float32)
    keep = _order_desc_lowest_index(gscore)[:, :topk_group]
    eligible = np.zeros((T, n_group), dtype=bool)
    np.put_along_axis(eligible, keep, True, axis=1)
    eligible = np.repeat(eligible, E // n_group, axis=1)
    masked = np.where(eligible, st, np.float32(-np.inf)).astype(np.float32)
    ids = _order_desc_lowest_index(masked)[:, :k].astype(np.int32)
    ssel = np.take_along_axis(s, ids, axis=1).astype(np.float64)
    gates = route_scale * ssel / ssel.sum(axis=1, keepdims=True)
    if return_groups:
        return ids, gates, keep.astype(np.int32), gscore
    return ids, gates


# ----------------------------------------------------------------------------
# Admission, count, prefix, permute  ([M6.2] 0x03B "Count, Prefix, Permute";
# [M6.6] 0x03B "Count, Prefix Sum, Permute"; [DISP] inverse bijection)
# ----------------------------------------------------------------------------

def permute(ids: np.ndarray, E: int, cap: int):
    """Stable expert-major permutation of accepted routes and its inverse.

    Route r = t*k + j carries expert ids[t, j].  Reading (admission order): a
    route is accepted iff fewer than ``cap`` earlier routes (in route id order)
    went to the same expert; cap < 0 means dropless.  Then
      c_e       = accepted routes of expert e,
      o_0 = 0,  o_{e+1} = o_e + c_e,
      pi        = accepted route ids ordered by (expert, route id)  (row -> route),
      pi_inv    = inverse of pi over accepted routes (route -> row, -1 if dropped).

    Returns dict(counts, offsets, row_to_route, route_to_row, n_dropped, ordinal).
    """
    e = np.asarray(ids, dtype=np.int64).reshape(-1)
    R = e.size
    if R and (e.min() < 0 or e.max() >= E):
        raise ValueError("expert id out of range")
    order = np.argsort(e, kind="stable")  # by (expert, route id)
    se = e[order]
    first = np.searchsorted(se, np.arange(E), side="left")
    ordinal = np.empty(R, dtype=np.int64)
    ordinal[order] = np.arange(R) - first[se]
    accepted = ordinal < cap if cap >= 0 else np.ones(R, dtype=bool)
    counts = np.bincount(e[accepted], minlength=E).astype(np.int64)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    route_to_row = np.full(R, -1, dtype=np.int64)
    route_to_row[accepted] = offsets[e[accepted]] + ordinal[accepted]
    row_to_route = np.empty(int(offsets[-1]), dtype=np.int64)
    acc_ids = np.nonzero(accepted)[0]
    row_to_route[route_to_row[acc_ids]] = acc_ids
    return dict(counts=counts, offsets=offsets, row_to_route=row_to_route,
                route_to_row=route_to_row, n_dropped=int(R - accepted.sum()), ordinal=ordinal)


def gather_rows(x_bits: np.ndarray, row_to_route: np.ndarray, k: int) -> np.ndarray:
    """x_perm[row] = x[token of route row_to_route[row]] (bit copy)."""
    return np.asarray(x_bits)[np.asarray(row_to_route) // k]


# ----------------------------------------------------------------------------
# SwiGLU expert  ([M6.6] 0x04A "The Frozen Six-Segment Input":
# E(X) = (SiLU(X Wg) * (X Wu)) W2, F = 6 n d d_ff; 0x04C "Variable Grouped GEMM")
# ----------------------------------------------------------------------------

def silu(g: np.ndarray) -> np.ndarray:
    # below g = -709 exp(-g) overflows to inf, and g / inf = -0.0 is SiLU's limit there
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


def swiglu(x_f64: np.ndarray, wg_f64: np.ndarray, wu_f64: np.ndarray, wd_f64: np.ndarray,
           round_h: bool = True, round_y: bool = True):
    """One expert on rows x [n,d] with weights Wg,Wu [d,I], Wd [I,d] (float64).

    Reading: H is stored as bf16 between the two products and y is returned
    as bf16 (the pages fix a BF16 returned row); accumulation is exact-ish in
    float64.  With round_* False the unrounded float64 values are returned.
    Returns (h, y) as float64 (bf16-valued when rounded).
    """
    g = x_f64 @ wg_f64
    u = x_f64 @ wu_f64
    h = silu(g) * u
    if round_h:
        h = bf16_to_f64(f64_to_bf16(h))
    y = h @ wd_f64
    if round_y:
        y = bf16_to_f64(f64_to_bf16(y))
    return h, y


def grouped_swiglu_rows(x_bits, seg_begin, seg_count, wg_bits, wu_bits, wd_bits, rows=None):
    """Grouped SwiGLU over row segments of x (bf16 bits); segment q uses expert q's weights.

    Returns (y_bits dict row -> bf16 bits [d], h_bits dict row -> bits [I]) for the
    requested ``rows`` (all segment rows if None).  Rows are grouped by segment
    so each expert's weights are converted once.
    """
    y_out, h_out = {}, {}
    for q, (b, c) in enumerate(zip(seg_begin, seg_count)):
        b, c = int(b), int(c)
        if c <= 0:
            continue
        rs = np.arange(b, b + c)
        if rows is not None:
            rs = np.intersect1d(rs, np.asarray(rows))
            if rs.size == 0:
                continue
        x = bf16_to_f64(np.asarray(x_bits)[rs])
        h, y = swiglu(x, bf16_to_f64(wg_bits[q]), bf16_to_f64(wu_bits[q]),
                      bf16_to_f64(wd_bits[q]))
        hb, yb = f64_to_bf16(h), f64_to_bf16(y)
        for i, r in enumerate(rs):
            y_out[int(r)] = yb[i]
            h_out[int(r)] = hb[i]
    return y_out, h_out


def swiglu_flops(rows: int, d: int, d_ff: int) -> int:
    """Matmul FLOPs of a SwiGLU expert over ``rows`` rows: 6 * rows * d * d_ff."""
    return 6 * rows * d * d_ff


# ----------------------------------------------------------------------------
# Combine  ([M6.6] 0x03C3 "Round-Trip Identity And Weighted Combine",
# 0x0CD; [M6.2] 0x03C "Forward Transpose Identity"; 0x0AE: gate applied once,
# after the expert, token accumulation in FP32)
# ----------------------------------------------------------------------------

def combine(y_rows_f64: np.ndarray, route_to_row: np.ndarray, gates: np.ndarray, T: int, k: int,
            shared_y_f64=None, out_init=None) -> np.ndarray:
    """out[t] = out_init[t] + sum over accepted slots j of gate[t,j] * y[row(t,j)] (+ shared[t]).

    Dropped routes (row -1) contribute nothing and the surviving gates are not
    renormalised.  The shared expert, when present, is added with weight one.
    Returns float64 [T, d].
    """
    r2r = np.asarray(route_to_row).reshape(T, k)
    g = np.asarray(gates, dtype=np.float64).reshape(T, k)
    d = y_rows_f64.shape[1]
    out = np.zeros((T, d)) if out_init is None else np.array(out_init, dtype=np.float64)
    for j in range(k):
        rows = r2r[:, j]
        ok = rows >= 0
        out[ok] += g[ok, j:j + 1] * y_rows_f64[rows[ok]]
    if shared_y_f64 is not None:
        out += shared_y_f64
    return out


def combine_token(y_lookup, route_to_row_t, gates_t, shared_t=None, init_t=None):
    """combine() for one token given a row -> y (float64 [d]) lookup."""
    acc = None if init_t is None else np.array(init_t, dtype=np.float64)
    for j, r in enumerate(route_to_row_t):
        if r < 0:
            continue
        term = float(gates_t[j]) * y_lookup(int(r))
        acc = term if acc is None else acc + term
    if shared_t is not None:
        acc = shared_t if acc is None else acc + shared_t
    return acc


# ----------------------------------------------------------------------------
# Pooled-wave layout  ([POOL] 02 "One pool for each destination GPU", 03 "Static
# shapes from send to combine", 04 "Capacity and memory", 05 "Carry expert IDs
# in-band", "Report both receiver rates", 07 "fixed source order")
# ----------------------------------------------------------------------------

def expert_to_dest_local(e, local_per_dest: int):
    """Expert e lives on destination e // L as local expert e % L (GPU 42 owns E252..E257)."""
    e = np.asarray(e)
    return e // local_per_dest, e % local_per_dest


def pool_pack(ids: np.ndarray, x_bits: np.ndarray, n_dest: int, local_per_dest: int,
              n_waves: int, pool_cap: int, wave: int, policy: str = "stripe"):
    """Sender side of one wave: fill the fixed per-destination pools.

    Routes to destination D are enumerated in route id order (ordinal j_D).
    Reading of the wave rule (policy):
      "stripe"  : wave = j_D mod n_waves, pool row = j_D div n_waves
      "destmod" : wave = D mod n_waves,   pool row = j_D
    A route of this wave whose row is >= pool_cap is a sender drop.  Pool
    row 0 is the header: element r < pool_cap holds the local expert id of
    payload row r (raw uint16 in the bf16 slot), EMPTY_HEADER if row r is
    unused; elements >= pool_cap are EMPTY_HEADER.  Payload row r is pool row
    1 + r, a bit copy of the token's activation row.  Unfilled payload rows
    are left zero here and are not part of the contract.

    Returns dict(pools uint16 [n_dest, pool_cap+1, d], route_to_poolrow int64 [R]
    (D*pool_cap + row, -1 when not placed in this wave), fill [n_dest],
    sender_drops (this wave), in_wave (bool [R])).
    """
    e = np.asarray(ids, dtype=np.int64).reshape(-1)
    R = e.size
    k = R // x_bits.shape[0]
    d = x_bits.shape[1]
    D, L = expert_to_dest_local(e, local_per_dest)
    order = np.argsort(D, kind="stable")
    sD = D[order]
    first = np.searchsorted(sD, np.arange(n_dest), side="left")
    jD = np.empty(R, dtype=np.int64)
    jD[order] = np.arange(R) - first[sD]
    if policy == "stripe":
        wv, row = jD % n_waves, jD // n_waves
    elif policy == "destmod":
        wv, row = D % n_waves, jD
    else:
        raise ValueError(policy)
    in_wave = wv == wave
    placed = in_wave & (row < pool_cap)
    pools = np.zeros((n_dest, pool_cap + 1, d), dtype=np.uint16)
    pools[:, 0, :] = EMPTY_HEADER
    pools[D[placed], 1 + row[placed]] = np.asarray(x_bits)[np.nonzero(placed)[0] // k]
    pools[D[placed], 0, row[placed]] = L[placed]
    route_to_poolrow = np.full(R, -1, dtype=np.int64)
    route_to_poolrow[placed] = D[placed] * pool_cap + row[placed]
    fill = np.bincount(D[placed], minlength=n_dest)
    return dict(pools=pools, route_to_poolrow=route_to_poolrow, fill=fill,
                sender_drops=int((in_wave & ~placed).sum()), in_wave=in_wave)


def pool_compact(pools: np.ndarray, pool_cap: int, n_local: int, local_cap: int,
                 first_source: int = 0):
    """Receiver side of one wave: group pooled rows into fixed per-local-expert arrays.

    Rows are visited in fixed source order (source pool ascending, then row);
    a row whose header id is l takes the next slot of local expert l, and is a
    receiver drop once that expert already holds local_cap rows.  Header ids
    that are neither < n_local nor EMPTY_HEADER are invalid and skipped.

    first_source > 0 is the per-receiver rotation [POOL] 07 mentions as a proposal
    (so overflow does not always fall on the same last sources).  Reading: the
    receiver visits sources first_source, first_source + 1, ..., n_src - 1, 0, ...,
    first_source - 1, each from row 0 up.

    Returns dict(compact uint16 [n_local, local_cap, d] (unfilled rows zero, not
    part of the contract), local_counts [n_local], poolrow_to_row int64
    [n_src*pool_cap] (l*local_cap + slot or -1, indexed by source*pool_cap + row),
    receiver_drops, bad_headers).
    """
    n_src, _, d = pools.shape
    if not 0 <= first_source < n_src:
        raise ValueError("first_source out of range")
    # visit position -> pool row (source * pool_cap + row)
    visit = (np.arange(n_src * pool_cap) // pool_cap + first_source) % n_src * pool_cap \
        + np.arange(n_src * pool_cap) % pool_cap
    flat = pools[:, 0, :pool_cap].astype(np.int64).reshape(-1)  # [n_src*pool_cap], src-major
    hdr = flat[visit]                                               # in visit order
    valid = hdr < n_local
    bad = int(((hdr != EMPTY_HEADER) & ~valid).sum())
    ordinal = np.full(hdr.size, -1, dtype=np.int64)
    vi = np.nonzero(valid)[0]
    lv = hdr[vi]
    order = np.argsort(lv, kind="stable")
    sl = lv[order]
    first = np.searchsorted(sl, np.arange(n_local), side="left")
    ov = np.empty(vi.size, dtype=np.int64)
    ov[order] = np.arange(vi.size) - first[sl]
    ordinal[vi] = ov
    keep = valid & (ordinal < local_cap) & (ordinal >= 0)
    poolrow_to_row = np.full(hdr.size, -1, dtype=np.int64)
    poolrow_to_row[visit[keep]] = hdr[keep] * local_cap + ordinal[keep]
    compact = np.zeros((n_local, local_cap, d), dtype=np.uint16)
    ki = np.nonzero(keep)[0]
    src, r = visit[ki] // pool_cap, visit[ki] % pool_cap
    compact[hdr[ki], ordinal[ki]] = pools[src, 1 + r]
    counts = np.minimum(np.bincount(hdr[vi], minlength=n_local), local_cap)
    return dict(compact=compact, local_counts=counts, poolrow_to_row=poolrow_to_row,
                receiver_drops=int(valid.sum() - keep.sum()), bad_headers=bad)


def compose_map(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """out[i] = b[a[i]] where a[i] >= 0, else -1 (route -> pool row -> compact row)."""
    a = np.asarray(a, dtype=np.int64)
    out = np.full(a.shape, -1, dtype=np.int64)
    ok = a >= 0
    out[ok] = np.asarray(b, dtype=np.int64)[a[ok]]
    return out


# ----------------------------------------------------------------------------
# Invariant checks of the maps  ([M6.6] 0x0CD "Route And Combine Assertions":
# accepted + dropped = routes, sum of counts = accepted, one inverse entry per
# accepted route; [M6.2] 0x03B stable order and inverse; [POOL] 02-05 headers,
# fills and one route per filled pool row).  Plain loops over every entry; they
# name each broken invariant so a one-field mutation can be traced to its check.
# ----------------------------------------------------------------------------

def expert_demand(ids: np.ndarray, E: int, live_routes: int = -1) -> np.ndarray:
    """n_e: routes among the first ``live_routes`` (all when < 0) that chose expert
    e, before any capacity ([M6.2] 0x01I).  Ids outside [0, E) are not counted."""
    e = np.asarray(ids, dtype=np.int64).reshape(-1)
    if live_routes >= 0:
        e = e[:live_routes]
    n = np.zeros(E, dtype=np.int64)
    for v in e:
        if 0 <= v < E:
            n[v] += 1
    return n


def permutation_violations(ids, E: int, cap: int, counts, offsets, row_to_route, route_to_row,
                           n_dropped: int, live_routes: int = -1) -> list:
    """Names of the permutation invariants that the given maps break ([] if none).

    row_to_route holds at least offsets[E] entries; route_to_row one per route.
    Routes at or past ``live_routes`` (padding slots of a token bucket) must map
    to -1.  Checked: offsets start at 0 and step by counts; counts are
    non-negative and (cap >= 0) at most cap; accepted + dropped = live routes and
    nothing is dropped when dropless; each accepted row points at a live route
    that points back, inside that route's expert segment; route ids increase
    along a segment; a dropped route's expert is full with routes of smaller id.
    """
    e = np.asarray(ids, dtype=np.int64).reshape(-1)
    R = e.size
    R_live = R if live_routes < 0 else min(R, max(live_routes, 0))
    counts = [int(v) for v in counts]
    offsets = [int(v) for v in offsets]
    r2r = [int(v) for v in route_to_row]
    row2 = [int(v) for v in row_to_route]
    bad = set()
    if offsets[0] != 0:
        bad.add("offsets[0]")
    for x in range(E):
        if counts[x] < 0 or offsets[x + 1] - offsets[x] != counts[x]:
            bad.add("offsets-counts")
        if cap >= 0 and counts[x] > cap:
            bad.add("capacity")
    acc = offsets[E]
    if acc < 0 or acc > R_live or acc + int(n_dropped) != R_live:
        bad.add("conservation")
    if cap < 0 and int(n_dropped) != 0:
        bad.add("dropless-drop")
    if acc < 0 or acc > R_live:
        return sorted(bad)
    for r in range(R):
        row = r2r[r]
        if r >= R_live:
            if row != -1:
                bad.add("padding-mapped")
            continue
        known = 0 <= e[r] < E
        if row >= 0:
            if not known or row >= acc or row2[row] != r or \
                    not offsets[e[r]] <= row < offsets[e[r] + 1]:
                bad.add("route-to-row")
        elif row == -1:
            if known:
                c, o = counts[e[r]], offsets[e[r] + 1]
                if cap < 0 or c != cap or (c > 0 and (o < 1 or o > acc or row2[o - 1] > r)):
                    bad.add("drop-admission")
        else:
            bad.add("route-to-row")
    for i in range(acc):
        r = row2[i]
        if not 0 <= r < R_live or r2r[r] != i:
            bad.add("row-to-route")
        elif i + 1 < acc and 0 <= e[r] < E and i + 1 < offsets[e[r] + 1] and row2[i + 1] <= r:
            bad.add("stable-order")
    return sorted(bad)


def pool_violations(ids, n_dest: int, local_per_dest: int, pool_cap: int, headers,
                    route_to_poolrow, fill) -> list:
    """Invariants of one wave's sender pools; headers is [n_dest, d] (pool row 0).

    Checked: 0 <= fill <= pool_cap; header element r < fill holds a local id,
    every other element EMPTY_HEADER; a placed route points at a filled row of
    its destination whose header holds its local id; every filled row has exactly
    one route, and the routes of a pool increase along its rows.
    """
    e = np.asarray(ids, dtype=np.int64).reshape(-1)
    hdr = np.asarray(headers).astype(np.int64)
    fill = [int(v) for v in fill]
    L = local_per_dest
    bad = set()
    for D in range(n_dest):
        f = fill[D]
        if not 0 <= f <= pool_cap:
            bad.add("fill")
            continue
        for r in range(hdr.shape[1]):
            if (r < f and not hdr[D, r] < L) or (r >= f and hdr[D, r] != EMPTY_HEADER):
                bad.add("header")
    owner = {}
    for r, p in enumerate(int(v) for v in route_to_poolrow):
        if p < 0:
            if p != -1:
                bad.add("route-to-poolrow")
            continue
        D, row = divmod(p, pool_cap)
        if not 0 <= e[r] < n_dest * L or D != e[r] // L or row >= fill[D] or \
                hdr[D, row] != e[r] % L or p in owner:
            bad.add("route-to-poolrow")
        owner.setdefault(p, r)
    for D in range(n_dest):
        f = min(fill[D], pool_cap)
        for row in range(pool_cap):
            p = D * pool_cap + row
            if row >= f:
                if p in owner:
                    bad.add("pool-row-owner")
            elif p not in owner or (row + 1 < f and owner.get(p + 1, -1) <= owner[p]):
                bad.add("pool-row-owner")
    return sorted(bad)


def compact_violations(headers, pool_cap: int, n_local: int, local_cap: int, local_counts,
                       poolrow_to_row, first_source: int = 0) -> list:
    """Invariants of one wave's receiver compact; headers is [n_src, >= pool_cap].

    Checked: 0 <= count <= local_cap; a pool row with a valid header l maps to
    -1 or to a slot of l below its count, any other row to -1; every slot below
    a count is the image of exactly one pool row and images keep the visiting
    order (sources from first_source on, rows ascending); a receiver drop's
    expert is full with rows that came earlier.
    """
    n_src = np.asarray(headers).shape[0]
    visit = (np.arange(n_src * pool_cap) // pool_cap + first_source) % n_src * pool_cap \
        + np.arange(n_src * pool_cap) % pool_cap
    flat_hdr = np.asarray(headers)[:, :pool_cap].astype(np.int64).reshape(-1)
    hdr = flat_hdr[visit]                              # in visit order
    cnt = [int(v) for v in local_counts]
    q_of = [int(v) for v in np.asarray(poolrow_to_row)[visit]]
    bad = set()
    for l in range(n_local):
        if not 0 <= cnt[l] <= local_cap:
            bad.add("local-count")
    owner = {}
    for i, q in enumerate(q_of):
        h = hdr[i]
        if q == -1:
            continue
        if not h < n_local or q < 0 or q // local_cap != h or q % local_cap >= cnt[h] or \
                q in owner:
            bad.add("poolrow-to-row")
        owner.setdefault(q, i)
    for i, q in enumerate(q_of):
        h = hdr[i]
        if h < n_local and q == -1:
            c = cnt[h]
            if c != local_cap or (c > 0 and owner.get(h * local_cap + c - 1, -1) > i):
                bad.add("receiver-drop")
    for l in range(n_local):
        f = min(cnt[l], local_cap)
        for slot in range(local_cap):
            q = l * local_cap + slot
            if slot >= f:
                if q in owner:
                    bad.add("slot-owner")
            elif q not in owner or (slot + 1 < f and owner.get(q + 1, -1) <= owner[q]):
                bad.add("slot-owner")
    return sorted(bad)


def drop_rates(total: int, sender: int, receiver: int):
    """[POOL] 05 'Report both receiver rates': S/T, R/T (additive) and R/(T-S)."""
    return dict(sender=sender / total, receiver=receiver / total,
                total=(sender + receiver) / total,
                receiver_conditional=(receiver / (total - sender)) if total > sender else 0.0)


# ----------------------------------------------------------------------------
# Backward of the transpose  ([M6.2] 0x03D "Backward Is The Reverse Semantic
# Transpose": Zbar_r = g_r * Ybar_origin(r), gbar_r = <Ybar_origin(r), Z_r>, and
# route-input gradients summed by origin token through the saved inverse)
# ----------------------------------------------------------------------------

def combine_backward(dout_f64: np.ndarray, y_rows_f64: np.ndarray, route_to_row: np.ndarray,
                     gates: np.ndarray, T: int, k: int):
    """Gradients of out[t] = sum_j g[t,j] * y[row(t,j)] for upstream dout [T, d].

    Returns (dy float64 [n_rows, d] -- g[t,j] * dout[t] on the row of every accepted
    route, zero elsewhere -- and dgates float64 [T, k] -- <dout[t], y[row(t,j)]>,
    zero for dropped routes).
    """
    r2r = np.asarray(route_to_row).reshape(T, k)
    g = np.asarray(gates, dtype=np.float64).reshape(T, k)
    dout = np.asarray(dout_f64, dtype=np.float64)
    dy = np.zeros_like(np.asarray(y_rows_f64, dtype=np.float64))
    dg = np.zeros((T, k))
    for j in range(k):
        rows = r2r[:, j]
        ok = rows >= 0
        dy[rows[ok]] = g[ok, j:j + 1] * dout[ok]
        dg[ok, j] = np.sum(dout[ok] * y_rows_f64[rows[ok]], axis=1)
    return dy, dg


def unpermute_grad(dx_perm_f64: np.ndarray, route_to_row: np.ndarray, T: int, k: int):
    """Token gradients: dx[t] = sum over the token's accepted routes of dx_perm[row(t,j)]."""
    r2r = np.asarray(route_to_row).reshape(T, k)
    d = dx_perm_f64.shape[1]
    dx = np.zeros((T, d))
    for j in range(k):
        rows = r2r[:, j]
        ok = rows >= 0
        dx[ok] += dx_perm_f64[rows[ok]]
    return dx


# ----------------------------------------------------------------------------
# Load telemetry and the loss-free bias step  ([M6.2] 0x01I skew summaries,
# 0x06E "The Bias Is A Delayed Controller State", 0x06J1-0x06J3)
# ----------------------------------------------------------------------------

def load_stats(counts) -> dict:
    """Skew summaries of a nonnegative count vector n over U units.

    mu = R / U; CV^2 = mean((n - mu)^2) / mu^2; rho_max = max(n) / mu;
    q = n / R with 0 log 0 = 0; H_norm = -sum q log q / log U; E_eff = exp(-sum q log q);
    MaxVio = (max(n) - mu) / mu.  Reading: an all-zero vector (R = 0) has all
    summaries 0, and H_norm is 0 when U = 1.
    """
    n = np.asarray(counts, dtype=np.float64)
    U = n.size
    R = n.sum()
    if U == 0 or R == 0:
        return dict(cv2=0.0, rho_max=0.0, h_norm=0.0, e_eff=0.0, max_vio=0.0, total=0)
    mu = R / U
    q = n / R
    with np.errstate(divide="ignore", invalid="ignore"):
        ent = -np.sum(np.where(q > 0, q * np.log(np.where(q > 0, q, 1.0)), 0.0))
    return dict(cv2=float(np.mean((n - mu) ** 2) / mu ** 2), rho_max=float(n.max() / mu),
                h_norm=float(ent / np.log(U)) if U > 1 else 0.0, e_eff=float(np.exp(ent)),
                max_vio=float((n.max() - mu) / mu), total=int(R))


def bias_update(bias, counts, u: float, rule: str = "sign") -> np.ndarray:
    """One delayed controller step on the fp32 selection bias.

    sign:         b_e <- b_e + u * sign(mean(c) - c_e)
    proportional: b_e <- b_e + u * (mean(c) - c_e)
    Reading: the increment is formed in float64 and rounded to fp32 once, then
    added to the fp32 bias with one fp32 rounding.
    """
    b = np.asarray(bias, dtype=np.float32)
    c = np.asarray(counts, dtype=np.float64)
    err = c.mean() - c
    step = np.sign(err) if rule == "sign" else err
    inc = (np.float64(np.float32(u)) * step).astype(np.float32)
    return (b + inc).astype(np.float32)


# ----------------------------------------------------------------------------
# FP8 dispatch payload with fp32 scales  ([M6.6] 0x0AB "Deriving BF16 And FP8
# Payloads", 0x0AC "Scale Tensor Ownership And Row Trace", 0x0AE "Router, Gate,
# Combine, And Accumulation Dtypes")
#
# Readings (the pages name "FP8" and fp32 scales, one per row or one per 128
# values of a row, but fix neither the FP8 format nor how a scale is chosen):
#   * format: E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; no
#     infinities; S.1111.111 is NaN; largest finite value 448);
#   * scale of a group: s = fp32(amax / 448), amax the largest |x| of the group
#     (exact), s = 1 for an all-zero group; groups are the whole row, or 128
#     consecutive values with a shorter last group when 128 does not divide d;
#   * code: q = E4M3(fp32(x / s)), rounded to nearest with ties to even and
#     saturated to +-448; the quotient is rounded to fp32 first, as a device
#     computes it;
#   * dequantized operand: xhat = bf16(fp32(decode(q) * s)), one fp32 rounding
#     of the exact product, then one bf16 rounding: the expert arithmetic that
#     follows is the bf16 path's.
# ----------------------------------------------------------------------------

E4M3_MAX = 448.0
E4M3_NAN = 0x7F


def e4m3_decode(codes) -> np.ndarray:
    """E4M3 codes (uint8) -> float64, from the format's definition."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    exp = (c >> 3) & 0xF
    man = (c & 0x7).astype(np.float64)
    mag = np.where(exp == 0, man / 8.0 * 2.0 ** -6, (1.0 + man / 8.0) * np.exp2(exp - 7.0))
    mag = np.where((exp == 15) & ((c & 0x7) == 7), np.nan, mag)
    return sign * mag


# the 127 finite non-negative E4M3 values in code order (code i has value _E4M3_POS[i])
_E4M3_POS = e4m3_decode(np.arange(0x7F, dtype=np.uint8))


def e4m3_encode(v) -> np.ndarray:
    """float values -> E4M3 codes: nearest finite value, ties to the even code,
    magnitudes above 448 saturate to 448, NaN -> 0x7F (sign kept), sign of zero kept."""
    v = np.asarray(v, dtype=np.float64)
    mag = np.abs(v)
    sat = np.minimum(mag, E4M3_MAX)
    hi = np.clip(np.searchsorted(_E4M3_POS, sat, side="left"), 0, 0x7E)  # first value >= sat
    lo = np.maximum(hi - 1, 0)
    d_lo = sat - _E4M3_POS[lo]
    d_hi = _E4M3_POS[hi] - sat
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(np.isnan(v), E4M3_NAN, code)
    neg = np.signbit(v)
    return (code | np.where(neg, 0x80, 0)).astype(np.uint8)


def n_scale_groups(d: int, group: int) -> int:
    """Scales per row: 1 for a whole-row scale (group 0), ceil(d / group) otherwise."""
    return 1 if group == 0 else -(-d // group)


def quantize_fp8(x_bits: np.ndarray, group: int):
    """bf16 rows [n, d] -> (E4M3 codes uint8 [n, d], fp32 scales [n, G]).

    group 0: one scale per row; group 128: one scale per 128 values of a row.
    """
    x = bf16_to_f64(np.asarray(x_bits)).astype(np.float32)  # exact
    n, d = x.shape
    g = d if group == 0 else group
    G = n_scale_groups(d, group)
    codes = np.empty((n, d), dtype=np.uint8)
    scales = np.empty((n, G), dtype=np.float32)
    for j in range(G):
        blk = x[:, j * g:(j + 1) * g]
        amax = np.abs(blk).max(axis=1) if blk.shape[1] else np.zeros(n, np.float32)
        s = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
        scales[:, j] = s
        quot = (blk / s[:, None]).astype(np.float32)  # IEEE fp32 division
        codes[:, j * g:(j + 1) * g] = e4m3_encode(quot)
    return codes, scales


def dequantize_fp8(codes: np.ndarray, scales: np.ndarray, group: int) -> np.ndarray:
    """(E4M3 codes [n, d], fp32 scales [n, G]) -> bf16 bits [n, d] of the dequantized rows."""
    c = np.asarray(codes)
    n, d = c.shape
    g = d if group == 0 else group
    s_full = np.repeat(np.asarray(scales, dtype=np.float64), g, axis=1)[:, :d]
    prod = e4m3_decode(c) * s_full          # exact in float64 (4 x 24 significant bits)
    return f64_to_bf16(prod.astype(np.float32).astype(np.float64))


def payload_bytes(rows: int, d: int, mode: str, group: int = 128) -> int:
    """Logical dispatch payload of `rows` routed rows of width d ([M6.6] 0x0AB):
    bf16: rows*d*2; fp8_row: rows*d + rows*4; fp8_block: rows*d + rows*ceil(d/group)*4."""
    if mode == "bf16":
        return rows * d * 2
    if mode == "fp8_row":
        return rows * d + rows * 4
    if mode == "fp8_block":
        return rows * d + rows * (-(-d // group)) * 4
    raise ValueError(mode)
