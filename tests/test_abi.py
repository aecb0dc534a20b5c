"""The C-ABI library: it builds for sm_103a, loads without a GPU, exports every
function include/moe.h declares, and rejects bad arguments on the host (these
calls return before any CUDA call, so they run without a GPU)."""
import ctypes
import subprocess

import pytest

from moe_token_routing_index_gb300 import build as mbuild


@pytest.fixture(scope="module")
def lib():
    mbuild.build()
    from moe_token_routing_index_gb300 import binding

    return binding


def test_library_exports_every_header_symbol(lib):
    names = lib.header_symbols()
    assert len(names) >= 13
    exported = subprocess.run(["nm", "-D", "--defined-only", str(lib.LIB_PATH)], capture_output=True,
                              text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in exported.splitlines() if ln.strip()}
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        assert hasattr(lib.library(), n)


def test_status_strings(lib):
    L = lib.library()
    assert L.moe_status_string(0) == b"ok"
    assert b"invalid" in L.moe_status_string(-1)
    assert b"workspace" in L.moe_status_string(-4)


def test_host_side_validation_without_gpu(lib):
    L = lib.library()
    n = ctypes.c_size_t(0)
    assert L.moe_route_workspace_size(-1, 8, 1, ctypes.byref(n)) == lib.MOE_ERR_INVALID
    assert L.moe_route_workspace_size(64, 8, 9, ctypes.byref(n)) == lib.MOE_ERR_INVALID      # top_k > E
    assert L.moe_route_workspace_size(64, 2048, 1, ctypes.byref(n)) == lib.MOE_ERR_UNSUPPORTED
    assert L.moe_route_workspace_size(64, 8, 2, ctypes.byref(n)) == lib.MOE_OK and n.value > 0
    fake = ctypes.c_void_p(0x1000)
    # route: workspace too small
    assert L.moe_route(fake, 0, 8, 1, 64, 8, 2, None, fake, fake, fake, fake, None, None, fake, 16, None) \
        == lib.MOE_ERR_WORKSPACE
    # route: null counts
    assert L.moe_route(fake, 0, 8, 1, 64, 8, 2, None, None, fake, fake, fake, None, None, fake, 1 << 20, None) \
        == lib.MOE_ERR_INVALID
    # gather: D not a multiple of 16; empty is a no-op
    assert L.moe_gather_scale(fake, 4, 24, fake, fake, 4, fake, 0, 8, 1, 8, None, None, 1, fake, None) \
        == lib.MOE_ERR_UNSUPPORTED
    assert L.moe_gather_scale(None, 4, 32, None, None, 0, None, 0, 8, 1, 8, None, None, 1, None, None) == lib.MOE_OK
    # gather: bad score dtype; inverse permutation without a valid top_k
    assert L.moe_gather_scale(fake, 4, 32, fake, fake, 4, fake, 7, 8, 1, 8, None, None, 1, fake, None) \
        == lib.MOE_ERR_INVALID
    assert L.moe_gather_scale(fake, 4, 32, fake, fake, 4, fake, 0, 8, 1, 8, None, fake, 0, fake, None) \
        == lib.MOE_ERR_INVALID
    # quantising gather needs out_scale
    assert L.moe_gather_scale_quant(fake, 4, 32, fake, fake, 4, fake, 0, 8, 1, 8, None, None, 1, None, fake, None,
                                    None) == lib.MOE_ERR_INVALID
    # scatter: top_k > 1 needs the inverse permutation
    assert L.moe_scatter_add(fake, fake, fake, None, 2, 8, 4, 32, None, 1, None) == lib.MOE_ERR_INVALID
    # silu: misaligned row stride
    assert L.moe_silu_mul(fake, fake, 36, 4, 32, None, fake, None) == lib.MOE_ERR_UNSUPPORTED
    # grouped GEMM: N not a multiple of 16, unknown epilogue, too many experts
    nq = (None, None, None)    # scale_ub, z_out, z_scale (the SILU_MUL_QUANT epilogue only)
    assert L.moe_grouped_gemm(fake, fake, fake, 4, 64, 24, 64, fake, 0, None, 0, 0, *nq, None) \
        == lib.MOE_ERR_UNSUPPORTED
    assert L.moe_grouped_gemm(fake, fake, fake, 4, 64, 32, 64, fake, 9, None, 0, 0, *nq, None) == lib.MOE_ERR_INVALID
    assert L.moe_grouped_gemm(fake, fake, fake, 2048, 64, 32, 64, fake, 0, None, 0, 0, *nq, None) \
        == lib.MOE_ERR_UNSUPPORTED
    assert L.moe_grouped_gemm_fp8_rowwise(fake, fake, fake, None, fake, 4, 64, 32, 64, fake, 0, None, 0, 0, *nq,
                                          None) == lib.MOE_ERR_INVALID
    # the fused combine only goes with the plain epilogue
    assert L.moe_grouped_gemm(fake, fake, fake, 4, 64, 32, 64, fake, 1, fake, 8, 1, *nq, None) == lib.MOE_ERR_INVALID
    # SILU_MUL_QUANT needs z_out and z_scale, a 16-byte aligned z_out and H <= 16384
    q = lib.MOE_EPILOGUE_SILU_MUL_QUANT
    assert L.moe_grouped_gemm(fake, fake, fake, 4, 64, 64, 64, fake, q, None, 0, 0, None, None, fake, None) \
        == lib.MOE_ERR_INVALID
    assert L.moe_grouped_gemm_fp8_rowwise(fake, fake, fake, fake, fake, 4, 64, 64, 64, fake, q, None, 0, 0, None,
                                          fake, None, None) == lib.MOE_ERR_INVALID
    assert L.moe_grouped_gemm(fake, fake, fake, 4, 64, 64, 64, fake, q, None, 0, 0, None, ctypes.c_void_p(0x1008),
                              fake, None) == lib.MOE_ERR_UNSUPPORTED
    assert L.moe_grouped_gemm(fake, fake, fake, 4, 64, 2 * 16400, 64, fake, q, None, 0, 0, None, fake, fake, None) \
        == lib.MOE_ERR_UNSUPPORTED
    assert L.moe_grouped_gemm(fake, fake, fake, 4, 64, 64, 64, fake, q, fake, 8, 1, None, fake, fake, None) \
        == lib.MOE_ERR_INVALID
    n = ctypes.c_size_t(0)
    assert L.moe_expert_mlp_workspace_size(0, ctypes.byref(n)) == lib.MOE_ERR_INVALID
    assert L.moe_expert_mlp(fake, fake, fake, fake, 4, 64, 32, 32, fake, fake, None, 0, 0, fake, 0, 0, None) \
        == lib.MOE_ERR_WORKSPACE
    # expert MLP: unknown flag bits; packed weights need H and D multiples of 128
    assert L.moe_expert_mlp(fake, fake, fake, fake, 4, 64, 128, 128, fake, fake, None, 0, 0, fake, 1 << 20, 0x400,
                            None) == lib.MOE_ERR_INVALID
    assert L.moe_expert_mlp(fake, fake, fake, fake, 4, 64, 128, 96, fake, fake, None, 0, 0, fake, 1 << 20,
                            lib.MOE_WEIGHTS_PACKED, None) == lib.MOE_ERR_UNSUPPORTED
    # packed weights: N (and its halves with SiLU*mul) a multiple of 128
    assert L.moe_grouped_gemm(fake, fake, fake, 4, 64, 96, 64, fake, lib.MOE_WEIGHTS_PACKED, None, 0, 0, *nq,
                              None) == lib.MOE_ERR_UNSUPPORTED
    assert L.moe_grouped_gemm(fake, fake, fake, 4, 64, 128, 64, fake, lib.MOE_WEIGHTS_PACKED | 1, None, 0, 0, *nq,
                              None) == lib.MOE_ERR_UNSUPPORTED                    # SiLU halves of 64 rows
    # pack size: bf16 [2, 256, 208] -> 4 row blocks x ceil(416 / 128) = 4 column blocks of 16 KB
    assert L.moe_pack_weights_size(2, 256, 208, lib.MOE_DTYPE_BF16, ctypes.byref(n)) == lib.MOE_OK
    assert n.value == 4 * 4 * 16384
    # e4m3 [3, 100, 256]: 300 rows -> 3 row blocks (zero rows past the end) x 2 column blocks
    assert L.moe_pack_weights_size(3, 100, 256, lib.MOE_DTYPE_E4M3, ctypes.byref(n)) == lib.MOE_OK
    assert n.value == 3 * 2 * 16384
    assert L.moe_pack_weights_size(2, 256, 208, lib.MOE_DTYPE_F32, ctypes.byref(n)) == lib.MOE_ERR_INVALID
    assert L.moe_pack_weights_size(2, 256, 24, lib.MOE_DTYPE_BF16, ctypes.byref(n)) == lib.MOE_ERR_UNSUPPORTED
    assert L.moe_pack_weights(None, 2, 256, 64, lib.MOE_DTYPE_BF16, fake, None) == lib.MOE_ERR_INVALID
    # router scores: shape limits, workspace, empty batch
    assert L.moe_router_workspace_size(-1, 64, 8, ctypes.byref(n)) == lib.MOE_ERR_INVALID
    assert L.moe_router_workspace_size(64, 64, 300, ctypes.byref(n)) == lib.MOE_ERR_UNSUPPORTED
    assert L.moe_router_workspace_size(64, 24, 8, ctypes.byref(n)) == lib.MOE_ERR_UNSUPPORTED
    assert L.moe_router_workspace_size(0, 64, 8, ctypes.byref(n)) == lib.MOE_OK and n.value == 0
    assert L.moe_router_workspace_size(8192, 5120, 16, ctypes.byref(n)) == lib.MOE_OK
    assert L.moe_router_scores(fake, 8192, 5120, fake, 0, None, fake, None, 0, None) == lib.MOE_ERR_INVALID
    assert L.moe_router_scores(fake, 8192, 5120, ctypes.c_void_p(0x1008), 16, None, fake, None, 0, None) \
        == lib.MOE_ERR_UNSUPPORTED                                                   # misaligned router weight
    assert L.moe_router_scores(None, 0, 64, None, 8, None, None, None, 0, None) == lib.MOE_OK
    assert L.moe_router_scores(None, 4, 64, fake, 8, None, fake, fake, 1 << 30, None) == lib.MOE_ERR_INVALID
    # top-k finalize: bad weight dtype, odd D, empty is a no-op
    assert L.moe_topk_finalize(fake, 8, 32, fake, 7, fake, 4, 2, None, None, fake, None) == lib.MOE_ERR_INVALID
    assert L.moe_topk_finalize(fake, 8, 24, fake, 1, fake, 4, 2, None, None, fake, None) == lib.MOE_ERR_UNSUPPORTED
    assert L.moe_topk_finalize(None, 0, 32, None, 1, None, 0, 2, None, None, None, None) == lib.MOE_OK
    assert L.moe_topk_finalize(fake, 8, 32, fake, 1, fake, 4, 0, None, None, fake, None) == lib.MOE_ERR_INVALID
    # padded scatter: T_K not a multiple of T, missing counts, top_k > 1 without the inverse permutation
    assert L.moe_scatter_add_padded(fake, fake, fake, 8, fake, None, 1, 30, 8, 32, 1, None) == lib.MOE_ERR_INVALID
    assert L.moe_scatter_add_padded(fake, fake, None, 8, fake, None, 1, 32, 8, 32, 1, None) == lib.MOE_ERR_INVALID
    assert L.moe_scatter_add_padded(fake, fake, fake, 8, fake, None, 2, 32, 16, 32, 1, None) == lib.MOE_ERR_INVALID
    # bounded-wait self-test: unknown mode, limits outside [1 us, 2 s]
    assert L.moe_selftest_bounded_wait(2, 1000000, None) == lib.MOE_ERR_INVALID
    assert L.moe_selftest_bounded_wait(0, 10, None) == lib.MOE_ERR_INVALID
    assert L.moe_selftest_bounded_wait(1, 3000000000, None) == lib.MOE_ERR_INVALID
