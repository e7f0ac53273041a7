"""The C-ABI library builds, loads and exports every entry point include/moe.h
declares; host-side argument validation rejects bad calls before any launch.
No GPU is touched: every call here returns before the first CUDA call.
"""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from grouped_expert_gemm_gb300 import build, abi
    build.build()
    return abi.lib()


def declared_symbols():
    with open(os.path.join(ROOT, "include", "moe.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for name in ["moe_route", "moe_permute", "moe_grouped_swiglu", "moe_combine", "moe_pool_pack",
                 "moe_pool_compact"]:
        assert name in syms


def test_library_exports_every_declared_symbol(lib):
    from grouped_expert_gemm_gb300 import abi
    for name in declared_symbols():
        assert hasattr(lib, name), name
    assert sorted(abi.EXPORTED) == declared_symbols()


def test_capacity(lib):
    from grouped_expert_gemm_gb300 import abi, capacity_from_factor
    assert abi.moe_capacity(5, 4, 512, 8) == 80
    assert capacity_from_factor(1.0, 8192 * 8, 256) == 256
    assert capacity_from_factor(1.10, 524288, 64 * 3) == 3004
    assert capacity_from_factor(1.15, 524288, 6 * 3) == 33497
    assert capacity_from_factor(1.1, 10, 1) == 11
    assert abi.moe_capacity(1, 0, 5, 5) == -1
    assert abi.moe_capacity(1, 1, 5, 0) == -1


def test_host_validation_rejects_before_launch(lib):
    from grouped_expert_gemm_gb300 import abi
    P = abi.RouteParams
    # k > E, E too large, unknown score function, bias with softmax
    assert lib.moe_route(P(4, 4, 5, 0, 1, 1, 1.0), 16, None, 16, 16, None, None) == abi.MOE_ERR_INVALID_ARG
    assert lib.moe_route(P(4, 1024, 2, 0, 1, 1, 1.0), 16, None, 16, 16, None, None) == abi.MOE_ERR_UNSUPPORTED
    assert lib.moe_route(P(4, 8, 2, 7, 1, 1, 1.0), 16, None, 16, 16, None, None) == abi.MOE_ERR_INVALID_ARG
    assert lib.moe_route(P(4, 8, 2, 0, 1, 1, 1.0), 16, 16, 16, 16, None, None) == abi.MOE_ERR_INVALID_ARG
    # grouped: E not divisible by n_group, too few eligible experts
    assert lib.moe_route(P(4, 10, 2, 1, 4, 2, 2.5), 16, None, 16, 16, None, None) == abi.MOE_ERR_INVALID_ARG
    assert lib.moe_route(P(4, 16, 8, 1, 4, 1, 2.5), 16, None, 16, 16, None, None) == abi.MOE_ERR_UNSUPPORTED
    assert lib.moe_route(P(0, 8, 2, 0, 1, 1, 1.0), None, None, None, None, None, None) == abi.MOE_OK
    # bucket staging: negative T, no count pointer, d not a multiple of 8, misaligned rows
    assert lib.moe_bucket_stage(-1, 8, 64, 16, 16, 16, 16, 16, None) == abi.MOE_ERR_INVALID_ARG
    assert lib.moe_bucket_stage(2, 8, 64, 16, 16, 16, 16, None, None) == abi.MOE_ERR_INVALID_ARG
    assert lib.moe_bucket_stage(2, 8, 64, None, 16, 16, 16, 16, None) == abi.MOE_ERR_INVALID_ARG
    assert lib.moe_bucket_stage(2, 8, 60, 16, 16, 16, 16, 16, None) == abi.MOE_ERR_UNSUPPORTED
    assert lib.moe_bucket_stage(2, 8, 64, 16, 24, 16, 16, 16, None) == abi.MOE_ERR_UNSUPPORTED
    # permute: d not a multiple of 8, workspace too small, misaligned x
    assert lib.moe_permute(4, 12, 8, 2, -1, 16, 16, 16, 16, 16, 16, 16, 16, 16, 1 << 20, None,
                           None) == abi.MOE_ERR_UNSUPPORTED
    assert lib.moe_permute(4, 16, 8, 2, -1, 16, 16, 16, 16, 16, 16, 16, 16, 16, 0, None,
                           None) == abi.MOE_ERR_WORKSPACE_TOO_SMALL
    assert lib.moe_permute(4, 16, 8, 2, -1, 16, 18, 16, 16, 16, 16, 16, 16, 16, 1 << 20, None,
                           None) == abi.MOE_ERR_UNSUPPORTED
    # grouped GEMM: d not a multiple of 64, too many segments, workspace too small
    assert lib.moe_grouped_swiglu(2, 96, 128, 8, 16, 16, 16, 16, 16, 16, 16, 16, 1 << 30, None,
                                  None) == abi.MOE_ERR_UNSUPPORTED
    assert lib.moe_grouped_swiglu(2000, 64, 128, 8, 16, 16, 16, 16, 16, 16, 16, 16, 1 << 30, None,
                                  None) == abi.MOE_ERR_UNSUPPORTED
    assert lib.moe_grouped_swiglu(2, 64, 128, 8, 16, 16, 16, 16, 16, 16, 16, 16, 64, None,
                                  None) == abi.MOE_ERR_WORKSPACE_TOO_SMALL
    # combine: k too large, misaligned output
    assert lib.moe_combine(4, 17, 64, 16, 8, 16, 16, None, 0, 16, None, None) == abi.MOE_ERR_UNSUPPORTED
    assert lib.moe_combine(4, 2, 64, 16, 8, 16, 16, None, 0, 20, None, None) == abi.MOE_ERR_UNSUPPORTED
    # pool: header must fit one row, wave out of range
    pp = abi.PoolParams(4, 2, 3, 100, 0)
    assert lib.moe_pool_pack(pp, 4, 64, 2, 0, 16, 16, 16, 16, 16, 16, 16, 1 << 20, None,
                             None) == abi.MOE_ERR_UNSUPPORTED
    pp = abi.PoolParams(4, 2, 3, 8, 0)
    assert lib.moe_pool_pack(pp, 4, 64, 2, 3, 16, 16, 16, 16, 16, 16, 16, 1 << 20, None,
                             None) == abi.MOE_ERR_INVALID_ARG
    assert lib.moe_pool_compact(4, 100, 64, 2, 8, 16, 16, 16, 16, 16, 16, 1 << 20, None,
                                None) == abi.MOE_ERR_UNSUPPORTED
    assert lib.moe_compose_map(-1, 16, 16, 4, 16, None, None) == abi.MOE_ERR_INVALID_ARG
    # demand: E beyond the router's limit, missing output
    assert lib.moe_expert_demand(4, 2, 1024, None, 16, 16, None, None) == abi.MOE_ERR_UNSUPPORTED
    assert lib.moe_expert_demand(4, 2, 8, None, 16, None, None, None) == abi.MOE_ERR_INVALID_ARG
    # validators: bad sizes, a missing status word, too small a workspace, header too wide
    assert lib.moe_validate_permutation(4, 8, 9, -1, None, 16, 16, 16, 16, 16, 16, 16,
                                        None) == abi.MOE_ERR_INVALID_ARG
    assert lib.moe_validate_permutation(4, 8, 2, -1, None, 16, 16, 16, 16, 16, 16, None,
                                        None) == abi.MOE_ERR_INVALID_ARG
    assert lib.moe_validate_permutation(4, 600, 2, -1, None, 16, 16, 16, 16, 16, 16, 16,
                                        None) == abi.MOE_ERR_UNSUPPORTED
    pp = abi.PoolParams(4, 2, 3, 8, 0)
    assert lib.moe_validate_pools(pp, 4, 64, 2, 16, 16, 16, 16, 16, 8, 16,
                                  None) == abi.MOE_ERR_WORKSPACE_TOO_SMALL
    assert lib.moe_validate_pools(abi.PoolParams(4, 2, 3, 100, 0), 4, 64, 2, 16, 16, 16, 16, 16,
                                  1 << 20, 16, None) == abi.MOE_ERR_UNSUPPORTED
    assert lib.moe_validate_compact(4, 8, 64, 2, 10, 0, 16, 16, 16, 16, 79, 16,
                                    None) == abi.MOE_ERR_WORKSPACE_TOO_SMALL
    assert lib.moe_validate_compact(4, 100, 64, 2, 10, 0, 16, 16, 16, 16, 1 << 20, 16,
                                    None) == abi.MOE_ERR_UNSUPPORTED
    assert lib.moe_validate_compact(4, 8, 64, 2, 10, 4, 16, 16, 16, 16, 1 << 20, 16,
                                    None) == abi.MOE_ERR_INVALID_ARG  # first_source >= n_src
    assert lib.moe_pool_compact_rotated(4, 8, 64, 2, 10, -1, 16, 16, 16, 16, 16, 16, 1 << 20,
                                        None, None) == abi.MOE_ERR_INVALID_ARG
    # the wait self-test: limit outside (0, 1 s], missing status word
    assert lib.moe_debug_wait_timeout(0, 16, None) == abi.MOE_ERR_INVALID_ARG
    assert lib.moe_debug_wait_timeout(2000000000, 16, None) == abi.MOE_ERR_INVALID_ARG
    assert lib.moe_debug_wait_timeout(1000, None, None) == abi.MOE_ERR_INVALID_ARG


def test_workspace_sizes_are_monotone(lib):
    from grouped_expert_gemm_gb300 import abi
    assert abi.moe_permute_workspace_size(8192, 8, 256) >= abi.moe_permute_workspace_size(256, 2, 8)
    assert abi.moe_grouped_swiglu_workspace_size(65536, 2048) >= 65536 * 2048 * 2
    pp = abi.PoolParams(64, 6, 3, 3004, 0)
    assert abi.moe_pool_pack_workspace_size(pp, 65536, 8) >= 64 * 4
    assert abi.moe_pool_compact_workspace_size(64, 3004, 6) >= 6 * 4
    assert abi.moe_validate_pools_workspace_size(pp) == 64 * 3004 * 4
    assert abi.moe_validate_compact_workspace_size(6, 33497) == 6 * 33497 * 4


def test_status_strings(lib):
    from grouped_expert_gemm_gb300 import abi
    assert lib.moe_status_string(abi.MOE_OK) == b"ok"
    assert b"workspace" in lib.moe_status_string(abi.MOE_ERR_WORKSPACE_TOO_SMALL)
