"""FP8 dispatch payload kernels ([M6.6] 0x0AB-0x0AC) against the CPU oracle,
through the C ABI: E4M3 codes and fp32 scales bit-exact, the dequantized bf16
operand bit-exact, the FP8 permute moving each row and its scales to the same
route row, and the gate/up GEMM whose loader dequantizes E4M3 tiles giving
exactly the bf16 GEMM's result on the dequantized rows."""
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
    import grouped_expert_gemm_gb300 as g
    return g


def status0():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def _rows(n, d, seed):
    """bf16 rows of mixed magnitude with the special rows the scale rule has:
    all zero, tiny, one outlier, negative zeros."""
    gen = torch.Generator(device=DEV).manual_seed(seed)
    x = torch.randn((n, d), generator=gen, device=DEV)
    x = x * torch.exp(2 * torch.randn((n, 1), generator=gen, device=DEV))
    if n >= 4:
        x[0] = 0
        x[1] *= 1e-30
        x[2, d // 2] = 3.0e4
        x[3, : d // 3] = -0.0
    return x.to(torch.bfloat16)


def _quantize(x, group):
    g = G()
    n, d = x.shape
    ng = g.fp8_scale_groups(d, group)
    q = torch.empty((n, d), dtype=torch.uint8, device=DEV)
    s = torch.empty((n, ng), dtype=torch.float32, device=DEV)
    st = status0()
    g.moe_quantize_fp8(n, d, group, x, q, s, st)
    return q, s, st


@pytest.mark.parametrize("group", [0, 128])
@pytest.mark.parametrize("n,d", [(300, 64), (257, 2048), (33, 208), (9, 7168), (1, 16)])
def test_quantize_and_dequantize_bit_exact(group, n, d):
    g = G()
    x = _rows(n, d, seed=n + d)
    q, s, st = _quantize(x, group)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rq, rs = oracle.quantize_fp8(bits(x), group)
    assert np.array_equal(host(s).view(np.uint32), rs.view(np.uint32))
    assert np.array_equal(host(q), rq)
    xd = torch.empty((n, d), dtype=torch.bfloat16, device=DEV)
    g.moe_dequantize_fp8(n, d, group, q, s, xd)
    torch.cuda.synchronize()
    assert np.array_equal(bits(xd), oracle.dequantize_fp8(rq, rs, group))


def test_quantize_reports_nonfinite_input():
    g = G()
    x = _rows(8, 256, seed=1)
    x[5, 17] = float("inf")
    _, _, st = _quantize(x, 128)
    torch.cuda.synchronize()
    assert int(st.item()) & g.MOE_DEV_NONFINITE_INPUT


@pytest.mark.parametrize("group", [0, 128])
@pytest.mark.parametrize("T,d,E,k,cap", [(256, 64, 8, 2, 80), (300, 2048, 128, 8, -1),
                                         (5000, 192, 32, 4, 600), (1, 16, 4, 4, -1),
                                         (2, 2048, 128, 8, 1)])  # 16 routes: copied by the rank block
def test_permute_fp8_moves_rows_and_scales_together(group, T, d, E, k, cap):
    g = G()
    rng = np.random.default_rng(T + d)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    x = _rows(T, d, seed=3)
    q, s, _ = _quantize(x, group)
    ng = s.shape[1]
    R = T * k
    q_perm = torch.zeros((R, d), dtype=torch.uint8, device=DEV)
    s_perm = torch.full((R, ng), -1.0, dtype=torch.float32, device=DEV)
    i32 = dict(dtype=torch.int32, device=DEV)
    counts, offsets = torch.empty(E, **i32), torch.empty(E + 1, **i32)
    r2r, inv, nd = torch.empty(R, **i32), torch.empty(R, **i32), torch.zeros(1, **i32)
    wsb = g.moe_permute_workspace_size(T, k, E)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    st = status0()
    g.moe_permute_fp8(T, d, E, k, cap, group, torch.from_numpy(ids).to(DEV), q, s, q_perm, s_perm,
                      counts, offsets, r2r, inv, nd, ws, wsb, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = oracle.permute(ids, E, cap)
    acc = int(ref["offsets"][-1])
    assert host(counts).tolist() == ref["counts"].tolist()
    assert host(offsets).tolist() == ref["offsets"].tolist()
    assert np.array_equal(host(r2r)[:acc], ref["row_to_route"])
    assert np.array_equal(host(inv), ref["route_to_row"])
    assert int(nd.item()) == ref["n_dropped"]
    rq, rs = oracle.quantize_fp8(bits(x), group)
    assert np.array_equal(host(q_perm)[:acc], oracle.gather_rows(rq, ref["row_to_route"], k))
    assert np.array_equal(host(s_perm)[:acc].view(np.uint32),
                          oracle.gather_rows(rs, ref["row_to_route"], k).view(np.uint32))
    assert np.all(host(s_perm)[acc:] == -1.0)  # rows past the accepted total untouched


def _gate_up_fp8_case(n_seg, d, I, counts, group, seed=0, begins=None):
    g = G()
    counts = np.asarray(counts, np.int32)
    if begins is None:
        begins = np.concatenate([[0], np.cumsum(counts)[:-1]]).astype(np.int32)
    begins = np.asarray(begins, np.int32)
    max_rows = max(int((begins + counts).max()), 1)
    w = workloads.scaled(workloads.tiny(), d=d, I=I, E=n_seg, seed=seed)
    wg, wu, _ = workloads.make_expert_weights(w, DEV, n_experts=n_seg)
    x = _rows(max_rows, d, seed=seed + 11)
    q, s, _ = _quantize(x, group)
    xd = torch.empty_like(x)
    g.moe_dequantize_fp8(max_rows, d, group, q, s, xd)
    sb, sc = torch.from_numpy(begins).to(DEV), torch.from_numpy(counts).to(DEV)
    h8 = torch.full((max_rows, I), 5.0, dtype=torch.bfloat16, device=DEV)
    h16 = torch.full((max_rows, I), 5.0, dtype=torch.bfloat16, device=DEV)
    st = status0()
    g.moe_grouped_gate_up_fp8(n_seg, d, I, max_rows, group, q, s, sb, sc, wg, wu, h8, st)
    g.moe_grouped_gate_up(n_seg, d, I, max_rows, xd, sb, sc, wg, wu, h16, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    # the loader's operand is exactly the dequantized rows: identical bits everywhere,
    # including the rows outside every segment (never written by either)
    assert torch.equal(h8.view(torch.int16), h16.view(torch.int16))
    # and the result is the SwiGLU of the dequantized rows (oracle, sampled rows)
    rows = np.concatenate([np.arange(b, b + c) for b, c in zip(begins, counts)])
    pick = np.sort(np.random.default_rng(seed).choice(rows, min(48, rows.size), replace=False))
    xq_deq = oracle.dequantize_fp8(host(q), host(s), group)
    assert np.array_equal(bits(xd), xq_deq)
    for r in pick:
        qi = int(np.nonzero((begins <= r) & (r < begins + counts))[0][0])
        gg = oracle.bf16_to_f64(xq_deq[r:r + 1]) @ oracle.bf16_to_f64(bits(wg[qi]))
        uu = oracle.bf16_to_f64(xq_deq[r:r + 1]) @ oracle.bf16_to_f64(bits(wu[qi]))
        ref_h = oracle.bf16_to_f64(oracle.f64_to_bf16(oracle.silu(gg) * uu))
        assert_float_parity(oracle.bf16_to_f64(bits(h8[r:r + 1])), ref_h, f"H row {r}")


@pytest.mark.parametrize("group", [0, 128])
@pytest.mark.parametrize("n_seg,d,I,counts", [
    (1, 64, 128, [128]),
    (4, 64, 128, [130, 0, 7, 300]),
    (3, 192, 256, [255, 256, 257]),     # two scale groups, the last one 64 wide
    (5, 256, 384, [1, 129, 0, 64, 200]),
    (2, 192, 192, [150, 170]),          # I not a multiple of 128: 2 x 64-column tiles
    (6, 1024, 512, [400, 10, 300, 0, 129, 77]),
    (8, 2048, 768, [700, 520, 1, 333, 640, 0, 257, 512]),  # several tiles per CTA
])
def test_gate_up_fp8_equals_bf16_gemm_on_dequantized_rows(group, n_seg, d, I, counts):
    _gate_up_fp8_case(n_seg, d, I, counts, group, seed=n_seg + d)


@pytest.mark.parametrize("group", [0, 128])
@pytest.mark.parametrize("d", [256, 192])
def test_gate_up_fp8_many_tiles_per_cta(group, d):
    """Decode-like shape: 128 experts with a few rows each, several single-CTA tiles
    per CTA (and an odd number of k-steps per tile for d = 192)."""
    counts = np.random.default_rng(d).integers(0, 16, 128)
    _gate_up_fp8_case(128, d, 768, counts, group, seed=d + group)


def test_gate_up_fp8_gapped_segments():
    _gate_up_fp8_case(3, 128, 256, [40, 0, 90], 128, seed=3, begins=[10, 60, 200])
