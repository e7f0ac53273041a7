"""The allocation-free permute entry point (moe_permute_noalloc) against moe_permute
and the oracle.

moe_permute_noalloc serves callers that cannot call cudaMalloc and have no
workspace to lend (an inference runtime's plugin hook that may only enqueue on
the stream it is given, a latency-critical loop where an allocation could
synchronise the device).  It keeps its scratch in a fixed device array of the
library, shared by every call, so the test makes two calls in a row on
different inputs and checks that each matches moe_permute on the same input
bit for bit (the bar for integer and byte outputs), and that each matches the
oracle's permutation.  The file is collected last so that a run stopping at
the first failure has run every other test already.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def lib():
    from grouped_expert_gemm_gb300 import abi, build
    build.build()
    return abi.lib()


def _outputs(T, d, E, k):
    R = max(T * k, 1)
    return dict(
        x_perm=torch.full((R, d), -3, dtype=torch.int16, device=DEV),
        counts=torch.full((E,), -9, dtype=torch.int32, device=DEV),
        offsets=torch.full((E + 1,), -9, dtype=torch.int32, device=DEV),
        row_to_route=torch.full((R,), -9, dtype=torch.int32, device=DEV),
        route_to_row=torch.full((R,), -9, dtype=torch.int32, device=DEV),
        n_dropped=torch.full((1,), -9, dtype=torch.int32, device=DEV),
        status=torch.zeros((1,), dtype=torch.int32, device=DEV))


def _call(lib, fn, T, d, E, k, cap, ids, x, o, ws=None):
    stream = torch.cuda.current_stream().cuda_stream
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    common = [T, d, E, k, cap, p(ids), p(x), p(o["x_perm"]), p(o["counts"]), p(o["offsets"]),
              p(o["row_to_route"]), p(o["route_to_row"]), p(o["n_dropped"])]
    if fn == "moe_permute":
        st = lib.moe_permute(*common, p(ws), ws.numel(), p(o["status"]), ctypes.c_void_p(stream))
    else:
        st = lib.moe_permute_noalloc(*common, p(o["status"]), ctypes.c_void_p(stream))
    assert st == 0, f"{fn} returned status {st}"


@pytest.mark.parametrize("T,d,E,k,cap", [(4096, 256, 128, 8, -1), (3000, 64, 256, 8, 100)])
def test_noalloc_matches_permute_on_two_calls_in_a_row(lib, T, d, E, k, cap):
    rng = np.random.default_rng(T + E)
    outs = []
    for call in range(2):
        p = rng.dirichlet(np.ones(E) * (0.3 + call))
        ids_np = np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)])
        ids = torch.from_numpy(ids_np.astype(np.int32)).to(DEV)
        x = torch.randint(-30000, 30000, (T, d), dtype=torch.int16, device=DEV)
        ref = _outputs(T, d, E, k)
        wsb = lib.moe_permute_workspace_size(T, k, E)
        ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
        _call(lib, "moe_permute", T, d, E, k, cap, ids, x, ref, ws)
        got = _outputs(T, d, E, k)
        _call(lib, "moe_permute_noalloc", T, d, E, k, cap, ids, x, got)
        torch.cuda.synchronize()
        acc = int(ref["offsets"][-1].item())
        for name in ("counts", "offsets", "n_dropped", "status"):
            assert torch.equal(got[name], ref[name]), name
        assert torch.equal(got["route_to_row"][: T * k], ref["route_to_row"][: T * k])
        assert torch.equal(got["row_to_route"][:acc], ref["row_to_route"][:acc])
        assert torch.equal(got["x_perm"][:acc], ref["x_perm"][:acc])
        # and the oracle's permutation of the same routes
        orc = oracle.permute(ids_np.astype(np.int32), E, cap)
        assert got["counts"].cpu().numpy().tolist() == orc["counts"].tolist()
        assert got["offsets"].cpu().numpy().tolist() == orc["offsets"].tolist()
        assert int(got["n_dropped"].item()) == orc["n_dropped"]
        assert np.array_equal(got["route_to_row"][: T * k].cpu().numpy(), orc["route_to_row"])
        assert np.array_equal(got["row_to_route"][:acc].cpu().numpy(), orc["row_to_route"])
        xb = x.cpu().numpy().view(np.uint16)
        assert np.array_equal(got["x_perm"][:acc].cpu().numpy().view(np.uint16),
                              oracle.gather_rows(xb, orc["row_to_route"], k))
        outs.append(got)
    # the second call really saw different routing (the shared scratch was reused)
    assert not torch.equal(outs[0]["counts"], outs[1]["counts"])


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    # T*k*E large enough that the per-tile histogram would not fit the 64 KiB array
    T, k, E = 400000, 16, 512
    assert lib.moe_permute_workspace_size(T, k, E) > (64 << 10)
    null = ctypes.c_void_p(16)
    st = lib.moe_permute_noalloc(T, 64, E, k, -1, null, null, null, null, null, null, null, null,
                                 None, None)
    assert st == 2  # MOE_ERR_UNSUPPORTED, before anything is enqueued
