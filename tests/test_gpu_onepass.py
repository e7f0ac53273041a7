"""Both expert passes in one persistent launch (moe_grouped_swiglu_onepass).

[M6.6] 0x04C: the gate/up pass H = bf16(SiLU(X Wg) * (X Wu)), then the down pass
y = bf16(H Wd), over the same ragged segment table.  The one-launch kernel deals the
gate/up tiles and then the down tiles to one CTA per SM; a down tile waits (bounded)
for its expert's H rows on counters in a caller-owned int32 array that every call
leaves at zero.  Checked here against the oracle (every row of H and y), against the
two-launch calls bit for bit, over repeated calls (the counters return to zero), and
on a shape outside the one-launch kernel's reach (the two launches are issued).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from moe_check import assert_float_parity, bits, host

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    from grouped_expert_gemm_gb300 import build
    build.build()


def G():
    import grouped_expert_gemm_gb300 as m
    return m


def _inputs(n_seg, d, I, counts, seed):
    counts = np.asarray(counts, np.int32)
    begins = np.concatenate([[0], np.cumsum(counts)[:-1]]).astype(np.int32)
    max_rows = max(int(counts.sum()), 1)
    w = workloads.scaled(workloads.tiny(), d=d, I=I, E=n_seg, seed=seed)
    gen = torch.Generator(device=DEV).manual_seed(seed + 7)
    x = torch.randn((max_rows, d), generator=gen, device=DEV).to(torch.bfloat16)
    wg, wu, wd = workloads.make_expert_weights(w, DEV, n_experts=n_seg)
    return begins, counts, max_rows, x, wg, wu, wd


def _onepass(n_seg, d, I, max_rows, x, begins, counts, wg, wu, wd, sync, calls=1):
    g = G()
    h = torch.full((max_rows, I), 3.0, dtype=torch.bfloat16, device=DEV)
    y = torch.full((max_rows, d), 7.0, dtype=torch.bfloat16, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    b = torch.from_numpy(begins).to(DEV)
    c = torch.from_numpy(counts).to(DEV)
    for _ in range(calls):
        g.moe_grouped_swiglu_onepass(n_seg, d, I, max_rows, x, b, c, wg, wu, wd, h, y, sync, st)
    torch.cuda.synchronize()
    assert int(host(st)[0]) == 0
    return h, y


def _separate(n_seg, d, I, max_rows, x, begins, counts, wg, wu, wd):
    g = G()
    h = torch.full((max_rows, I), 3.0, dtype=torch.bfloat16, device=DEV)
    y = torch.full((max_rows, d), 7.0, dtype=torch.bfloat16, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    b = torch.from_numpy(begins).to(DEV)
    c = torch.from_numpy(counts).to(DEV)
    g.moe_grouped_gate_up(n_seg, d, I, max_rows, x, b, c, wg, wu, h, st)
    g.moe_grouped_down(n_seg, I, d, max_rows, h, b, c, wd, y, st)
    torch.cuda.synchronize()
    assert int(host(st)[0]) == 0
    return h, y


_R = np.random.default_rng(9)
CASES = [
    # (n_seg, d, I, counts, one launch taken)
    (128, 2048, 768, [1 if e % 16 == 3 else 0 for e in range(128)], True),   # one-token decode
    (128, 2048, 768, [1 if e % 4 == 1 else 0 for e in range(128)], True),    # four tokens
    (32, 1024, 768, [20 if e % 11 == 3 else e % 2 for e in range(32)], True),  # 2 m-blocks
    (32, 256, 768, list(_R.integers(1, 4, size=32)), True),                  # ~3 units per CTA
    (16, 4096, 512, [3, 0, 1, 0, 2, 5, 0, 1, 0, 0, 4, 1, 0, 2, 0, 1], True),   # 32 gate/up k-steps
    (128, 2048, 768, [1 if e % 8 == 5 else 0 for e in range(128)], False),   # two tokens: wide tiles
]


@pytest.mark.parametrize("n_seg,d,I,counts,taken", CASES)
def test_onepass_matches_the_oracle_and_the_two_launches(n_seg, d, I, counts, taken):
    begins, counts, max_rows, x, wg, wu, wd = _inputs(n_seg, d, I, counts, seed=n_seg + d)
    assert G().moe_grouped_swiglu_onepass_taken(n_seg, d, I, max_rows) == taken
    sync = torch.zeros(2 * n_seg, dtype=torch.int32, device=DEV)
    h, y = _onepass(n_seg, d, I, max_rows, x, begins, counts, wg, wu, wd, sync)
    assert int(sync.abs().sum()) == 0  # the counters are back at zero (or untouched)
    yr, hr = oracle.grouped_swiglu_rows(bits(x), begins, counts, bits(wg), bits(wu), bits(wd))
    rows = sorted(yr)
    assert_float_parity(oracle.bf16_to_f64(bits(h)[rows]),
                        oracle.bf16_to_f64(np.stack([hr[r] for r in rows])), "H")
    assert_float_parity(oracle.bf16_to_f64(bits(y)[rows]),
                        oracle.bf16_to_f64(np.stack([yr[r] for r in rows])), "y")
    hs, ys = _separate(n_seg, d, I, max_rows, x, begins, counts, wg, wu, wd)
    assert torch.equal(h[rows].view(torch.int16), hs[rows].view(torch.int16))
    assert torch.equal(y[rows].view(torch.int16), ys[rows].view(torch.int16))
    # rows outside every segment are never written
    untouched = np.setdiff1d(np.arange(max_rows), rows)
    assert bool((y[untouched] == 7.0).all())


def test_onepass_repeated_calls_leave_the_counters_at_zero():
    n_seg, d, I, counts, _ = CASES[0]
    begins, counts, max_rows, x, wg, wu, wd = _inputs(n_seg, d, I, counts, seed=5)
    sync = torch.zeros(2 * n_seg, dtype=torch.int32, device=DEV)
    h1, y1 = _onepass(n_seg, d, I, max_rows, x, begins, counts, wg, wu, wd, sync)
    h5, y5 = _onepass(n_seg, d, I, max_rows, x, begins, counts, wg, wu, wd, sync, calls=5)
    assert int(sync.abs().sum()) == 0
    assert torch.equal(y1.view(torch.int16), y5.view(torch.int16))
    assert torch.equal(h1.view(torch.int16), h5.view(torch.int16))


def test_onepass_outside_its_reach_issues_the_two_launches():
    """d = 192 is not a multiple of 128: the call runs the two passes and leaves sync alone."""
    n_seg, d, I, counts = 8, 192, 128, [3, 0, 5, 1, 0, 2, 7, 4]
    begins, counts, max_rows, x, wg, wu, wd = _inputs(n_seg, d, I, counts, seed=3)
    sync = torch.full((2 * n_seg,), 9, dtype=torch.int32, device=DEV)
    h, y = _onepass(n_seg, d, I, max_rows, x, begins, counts, wg, wu, wd, sync)
    assert bool((sync == 9).all())
    hs, ys = _separate(n_seg, d, I, max_rows, x, begins, counts, wg, wu, wd)
    rows = np.concatenate([np.arange(b, b + c) for b, c in zip(begins, counts)])
    assert torch.equal(y[rows].view(torch.int16), ys[rows].view(torch.int16))


@pytest.mark.parametrize("T", [1, 2, 4, 8])
def test_layer_with_one_launch_expert_passes_matches_the_two_launches(T):
    """The decode layer with expert_passes='onepass' against the same layer with the two
    launches (the oracle-checked layer path), bit for bit."""
    g = G()
    w = workloads.decode(T)
    logits, sel_bias = workloads.make_router_inputs(w, DEV)
    x = workloads.make_activations(w, DEV)
    wg, wu, wd = workloads.make_expert_weights(w, DEV)
    outs = []
    for passes in ("separate", "onepass"):
        layer = g.MoELayer(w.T, w.d, w.E, w.k, w.I, wg, wu, wd, expert_passes=passes, device=DEV)
        out = layer.forward(logits, x).clone()
        torch.cuda.synchronize()
        assert int(layer.dev_status.item()) == 0
        outs.append(out)
        if passes == "onepass":
            assert int(layer.onepass_sync.abs().sum()) == 0
    assert torch.equal(outs[0].view(torch.int32), outs[1].view(torch.int32))
