"""Decode graphs over a fixed token bucket ([M6.6] 0x05C-0x05F): padding slots are
masked before they get expert identities, a replay gives the real tokens the
oracle's routes, maps and outputs (and exactly the eager layer's bits), and the
exact admission predicate falls back to the eager layer without changing the
result."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from moe_check import (assert_float_parity, assert_gates, bits, host, oracle_token_outputs,
                       weights_fetcher)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    from grouped_expert_gemm_gb300 import build
    build.build()


@pytest.fixture(scope="module")
def weights():
    return workloads.make_expert_weights(workloads.decode(128), DEV)


@pytest.fixture(scope="module")
def bucket(weights):
    import grouped_expert_gemm_gb300 as g
    w = workloads.decode(128)
    wg, wu, wd = weights
    b = g.DecodeBucket(128, w.d, w.E, w.k, w.I, wg, wu, wd, device=DEV)
    b.capture()
    return b


@pytest.fixture(scope="module")
def ladder(weights):
    import grouped_expert_gemm_gb300 as g
    w = workloads.decode(128)
    wg, wu, wd = weights
    lad = g.DecodeBucketLadder([1, 2, 4, 8, 16, 32, 64, 128], w.d, w.E, w.k, w.I, wg, wu, wd,
                               device=DEV)
    lad.capture()
    return lad


@pytest.mark.parametrize("form", ["bucket", "ladder"])
@pytest.mark.parametrize("T", [1, 3, 5, 37, 128])
def test_replay_matches_the_oracle(request, weights, form, T):
    """A replay against the oracle on the decode workload's own inputs: the real
    tokens' ids, gates, counts, offsets and both maps (bit-exact or to the gate
    tolerance), every expert row y and the real tokens' output; padding slots keep
    masked ids, zero gates, -1 maps and zero output."""
    import grouped_expert_gemm_gb300 as g
    runner = request.getfixturevalue(form)
    w = workloads.decode(T)
    logits, _ = workloads.make_router_inputs(w, DEV)
    x = workloads.make_activations(w, DEV)
    out, path = runner.forward(logits, x)
    torch.cuda.synchronize()
    served = runner if form == "bucket" else runner.pick(T)
    assert path == ("replay" if form == "bucket" else f"replay:{served.B}")
    L, B, k = served.layer, served.B, w.k
    assert int(L.dev_status.item()) == 0
    ids, gates = oracle.route_softmax(host(logits), k)
    perm = oracle.permute(ids, w.E, -1)
    acc = int(perm["offsets"][-1])
    assert np.array_equal(host(L.topk_ids)[:T], ids)
    assert_gates(host(L.gates)[:T], gates)
    assert np.array_equal(host(L.counts), perm["counts"])
    assert np.array_equal(host(L.offsets), perm["offsets"])
    assert np.array_equal(host(L.row_to_route)[:acc], perm["row_to_route"])
    assert np.array_equal(host(L.route_to_row)[: T * k], perm["route_to_row"])
    assert int(L.n_dropped.item()) == 0
    # padding slots
    assert np.all(host(L.topk_ids)[T:] == g.MOE_ROUTE_MASKED)
    assert np.all(host(L.gates)[T:] == 0)
    assert np.all(host(L.route_to_row)[T * k: B * k] == -1)
    assert np.all(host(L.out)[T:] == 0)
    # expert rows and the real tokens' output
    xb = bits(x)
    ref_out, y_of_row = oracle_token_outputs(w, np.arange(T), xb, ids, gates, perm,
                                             weights_fetcher(*weights))
    yrows = np.array(sorted(y_of_row))
    assert yrows.size == acc
    got_y = oracle.bf16_to_f64(bits(L.y[torch.from_numpy(yrows).to(DEV)]))
    assert_float_parity(got_y, np.stack([y_of_row[r] for r in yrows]), "bucket replay y")
    assert_float_parity(host(out), ref_out, "bucket replay output")


def _inputs(T, seed, E=128, d=2048):
    gen = torch.Generator(device=DEV).manual_seed(seed)
    logits = torch.randn((T, E), generator=gen, device=DEV)
    x = torch.randn((T, d), generator=gen, device=DEV).to(torch.bfloat16)
    return logits, x


@pytest.mark.parametrize("T", [1, 37, 128, 5])
def test_replay_equals_eager_on_the_real_tokens(bucket, T):
    import grouped_expert_gemm_gb300 as g
    logits, x = _inputs(T, seed=T)
    out, path = bucket.forward(logits, x)
    torch.cuda.synchronize()
    assert path == "replay"
    L = bucket.layer
    assert int(L.dev_status.item()) == 0
    eager = g.MoELayer(T, **bucket.cfg, decode_path="separate")  # the 128-slot bucket's path
    ref = eager.forward(logits, x)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)  # same routes, rows, tiles: identical bits
    # padding slots never acquired expert identities or output
    k = bucket.k
    assert torch.all(L.topk_ids[T:] == g.MOE_ROUTE_MASKED)
    assert torch.all(L.gates[T:] == 0)
    assert torch.all(L.route_to_row[T * k:] == -1)
    assert int(L.counts.sum().item()) == T * k == int(L.offsets[-1].item())
    assert int(L.n_dropped.item()) == 0
    assert torch.all(L.out[T:] == 0)
    assert torch.equal(L.route_to_row[: T * k], eager.route_to_row[: T * k])


def test_replay_on_a_side_stream_with_inputs_to_convert(bucket):
    """Inputs that need conversion (fp16 logits, non-contiguous bf16 rows) written on
    the current stream, the step on another stream: the conversions wait for the
    writes and the replay gives the eager layer's bits."""
    import grouped_expert_gemm_gb300 as g
    T = 37
    logits, x = _inputs(T, seed=77)
    side = torch.cuda.Stream(DEV)
    for _ in range(3):  # each time on freshly written inputs
        lg16 = torch.empty((T, bucket.E), dtype=torch.float16, device=DEV)
        xt = torch.empty((bucket.d, T), dtype=torch.bfloat16, device=DEV)
        torch.cuda._sleep(2_000_000)  # the writes land well after the step is enqueued
        lg16.copy_(logits)
        xt.copy_(x.t())
        out, path = bucket.forward(lg16, xt.t(), stream=side)
        assert path == "replay"
        torch.cuda.current_stream().wait_stream(side)
        got = out.clone()
        torch.cuda.synchronize()
        ref = g.MoELayer(T, **bucket.cfg).forward(lg16.float(), xt.t().contiguous())
        torch.cuda.synchronize()
        assert torch.equal(got, ref)


def test_bucket_rejects_misshapen_inputs(bucket):
    logits, x = _inputs(4, seed=3)
    with pytest.raises(ValueError):
        bucket.forward(logits[:, :64], x)
    with pytest.raises(ValueError):
        bucket.forward(logits, x[:3])


def test_exact_admission_and_fallback(bucket):
    import grouped_expert_gemm_gb300 as g
    logits, x = _inputs(129, seed=9)
    out, path = bucket.forward(logits, x)
    assert path == "token_capacity_exceeded"
    ref = g.MoELayer(129, **bucket.cfg).forward(logits, x)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    small_l, small_x = _inputs(16, seed=10)
    assert bucket.forward(small_l, small_x, phase="prefill")[1] == "phase_not_decode"
    other = bucket.key[:4] + (bucket.key[4] + 1,) + bucket.key[5:]
    assert bucket.forward(small_l, small_x, key=other)[1] == "graph_key_mismatch"
    assert bucket.forward(small_l, small_x, key=bucket.key)[1] == "replay"


@pytest.mark.parametrize("cap", [-1, 3])
def test_permute_bucket_parity(cap):
    import grouped_expert_gemm_gb300 as g
    T, valid, d, E, k = 300, 211, 64, 32, 4
    rng = np.random.default_rng(cap + 5)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    ids[valid:] = 99999  # padding ids are garbage and must never be read
    x = torch.randn((T, d), device=DEV).to(torch.bfloat16)
    R = T * k
    outs = dict(x_perm=torch.zeros((R, d), dtype=torch.bfloat16, device=DEV),
                counts=torch.empty(E, dtype=torch.int32, device=DEV),
                offsets=torch.empty(E + 1, dtype=torch.int32, device=DEV),
                r2r=torch.full((R,), -5, dtype=torch.int32, device=DEV),
                inv=torch.full((R,), -5, dtype=torch.int32, device=DEV),
                nd=torch.zeros(1, dtype=torch.int32, device=DEV))
    wsb = g.moe_permute_workspace_size(T, k, E)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    vt = torch.tensor([valid], dtype=torch.int32, device=DEV)
    g.moe_permute_bucket(T, d, E, k, cap, vt, torch.from_numpy(ids).to(DEV), x, outs["x_perm"],
                         outs["counts"], outs["offsets"], outs["r2r"], outs["inv"], outs["nd"],
                         ws, wsb, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0  # the garbage ids were never read
    ref = oracle.permute(ids[:valid], E, cap)
    acc = int(ref["offsets"][-1])
    assert host(outs["counts"]).tolist() == ref["counts"].tolist()
    assert host(outs["offsets"]).tolist() == ref["offsets"].tolist()
    assert np.array_equal(host(outs["r2r"])[:acc], ref["row_to_route"])
    inv = host(outs["inv"])
    assert np.array_equal(inv[: valid * k], ref["route_to_row"])
    assert np.all(inv[valid * k:] == -1)
    assert int(outs["nd"].item()) == ref["n_dropped"]
    assert np.array_equal(bits(outs["x_perm"])[:acc],
                          oracle.gather_rows(bits(x), ref["row_to_route"], k))


@pytest.mark.parametrize("T,E,d", [(1, 128, 2048), (37, 128, 2048), (5, 7, 64), (0, 8, 64)])
def test_bucket_stage_copies_the_inputs_and_the_count(T, E, d):
    """One launch copies logits [T, E] and x [T, d] into the first T rows of the stable
    buffers, bit for bit, writes the count, and leaves the other rows alone."""
    import grouped_expert_gemm_gb300 as g
    B = 40 if T <= 40 else T
    gen = torch.Generator(device=DEV).manual_seed(T + E)
    logits = torch.randn((T, E), generator=gen, device=DEV)
    x = torch.randn((T, d), generator=gen, device=DEV).to(torch.bfloat16)
    ldst = torch.full((B, E), -3.0, device=DEV)
    xdst = torch.full((B, d), 5.0, dtype=torch.bfloat16, device=DEV)
    valid = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    g.moe_bucket_stage(T, E, d, logits, x, ldst, xdst, valid)
    torch.cuda.synchronize()
    assert int(valid.item()) == T
    assert torch.equal(ldst[:T], logits) and bool((ldst[T:] == -3.0).all())
    assert torch.equal(xdst[:T].view(torch.int16), x.view(torch.int16))
    assert bool((xdst[T:] == 5.0).all())


def test_ladder_replays_the_smallest_bucket_bit_identical_to_eager():
    """A ladder of buckets: each step replays the smallest bucket holding its tokens,
    with the eager layer's bits; above the largest bucket it falls back."""
    import grouped_expert_gemm_gb300 as g
    w = workloads.decode(128)
    wg, wu, wd = workloads.make_expert_weights(w, DEV)
    ladder = g.DecodeBucketLadder([1, 4, 16], w.d, w.E, w.k, w.I, wg, wu, wd, device=DEV)
    ladder.capture()
    for T, want in [(1, "replay:1"), (3, "replay:4"), (4, "replay:4"), (11, "replay:16"),
                    (17, "token_capacity_exceeded")]:
        logits, x = _inputs(T, seed=100 + T)
        out, path = ladder.forward(logits, x)
        ref = g.MoELayer(T, **ladder.buckets[0].cfg).forward(logits, x)
        torch.cuda.synchronize()
        assert path == want, (T, path)
        assert torch.equal(out, ref), T
    assert ladder.pick(16).B == 16 and ladder.pick(17) is None
