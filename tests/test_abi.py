"""CPU-side checks of the C ABI: the library builds, loads, exports every function that
include/moe.h declares, and its host-only calls (sizes, argument checks) behave."""
import ctypes
import os
import re

import pytest

import combine_moe_route_softmax_gb300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    with open(os.path.join(ROOT, "include", "moe.h")) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:[\w\s\*]+?)\b(moe_\w+)\s*\(", src, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(moe.LIB_PATH):
        from combine_moe_route_softmax_gb300 import build
        build.build()
    return moe.lib()


def test_header_declares_the_layer_calls():
    names = declared_functions()
    for n in ("moe_route_topk", "moe_permute", "moe_grouped_gemm", "moe_combine", "moe_layer_forward",
              "moe_permute_workspace_bytes", "moe_layer_workspace_bytes", "moe_combine_verify"):
        assert n in names


def test_library_exports_every_declared_function(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in moe._SIGS, f"binding has no signature for {name}"


def test_host_only_calls(lib):
    assert lib.moe_abi_version() == 6
    assert lib.moe_status_string(2) == b"workspace too small"
    # scratch sized from the inputs: grows with T, K and E
    a = lib.moe_permute_workspace_bytes(128, 8, 256, 1)
    b = lib.moe_permute_workspace_bytes(16384, 8, 256, 1)
    assert 0 < a < b and b % 256 == 0
    assert lib.moe_permute_workspace_bytes(16, 2, 0, 0) == 0
    # the batched layout keeps its cu_seqlens in the scratch: one more 256-byte-aligned region
    c = lib.moe_permute_batched_workspace_bytes(128, 8, 256, 1)
    assert c == a + 1280 and lib.moe_permute_batched_workspace_bytes(16, 2, 0, 0) == 0


def test_layer_workspace_size(lib):
    d = moe.LayerDesc(16384, 7168, 2048, 256, 8, moe.MOE_BF16, 1)
    n = lib.moe_layer_workspace_bytes(ctypes.byref(d))
    cap = 16384 * 8 + 16384
    assert n >= cap * 7168 * 2 * 2 + cap * 2048 * 2
    bad = moe.LayerDesc(16, 100, 2048, 8, 2, moe.MOE_BF16, 0)   # H not a multiple of 128
    assert lib.moe_layer_workspace_bytes(ctypes.byref(bad)) == 0
    # batched layout: (E + 1) blocks of max_tokens rows instead of T*K + T rows
    db = moe.LayerDesc(128, 7168, 2048, 256, 8, moe.MOE_E4M3, 1, 0, 128)
    nb = lib.moe_layer_workspace_bytes(ctypes.byref(db))
    assert nb >= 257 * 128 * (7168 + 2048 + 7168 * 2)
    views = moe.LayerViews()
    assert lib.moe_layer_views(ctypes.byref(db), 1 << 20, ctypes.byref(views)) == 0
    assert views.cap == 257 * 128 and views.cu_seqlens is None and views.masked_m == 1 << 20
    # fused combine: one more region, the [T, H/128] counters
    df = moe.LayerDesc(128, 7168, 2048, 256, 8, moe.MOE_E4M3, 1, 0, 0, 1)
    d0 = moe.LayerDesc(128, 7168, 2048, 256, 8, moe.MOE_E4M3, 1, 0, 0, 0)
    assert lib.moe_layer_workspace_bytes(ctypes.byref(df)) == lib.moe_layer_workspace_bytes(ctypes.byref(d0)) + \
        128 * 56 * 4
    assert lib.moe_layer_views(ctypes.byref(df), 1 << 20, ctypes.byref(views)) == 0 and views.counters
    df.fuse_combine = 2
    assert lib.moe_layer_workspace_bytes(ctypes.byref(df)) == 0
    # the combine fake-quant format is 0 (E4M3) or 1 (NVFP4); it does not change the workspace
    n0 = lib.moe_layer_workspace_bytes(ctypes.byref(d0))
    d0.combine_fq_format = 1
    assert lib.moe_layer_workspace_bytes(ctypes.byref(d0)) == n0 > 0
    d0.combine_fq_format = 2
    assert lib.moe_layer_workspace_bytes(ctypes.byref(d0)) == 0
    db.max_tokens = -1
    assert lib.moe_layer_workspace_bytes(ctypes.byref(db)) == 0
    db.max_tokens = 1 << 24   # 257 blocks of 2^24 rows: more than 2^31 rows
    assert lib.moe_layer_workspace_bytes(ctypes.byref(db)) == 0


def test_argument_errors_launch_nothing(lib):
    # K > E, and H % 128 != 0, are rejected on the host before any CUDA call
    assert lib.moe_route_topk(None, 4, 2, 3, None, None, None, None) == 1
    assert lib.moe_permute(None, 4, 2, 8, 0, None, 100, 0, None, None, None, None, None, None, None, 0, None,
                           None) == 1
    assert lib.moe_grouped_gemm(None, None, None, 1, 16, 100, 256, None, None, 1, None, None, 0, 0, None, None,
                                None, None) == 1
    assert lib.moe_combine(None, None, None, 4, 2, 100, None, None, None, None, None) == 1
    # NVFP4 combine: H not a multiple of 128, or no per-tensor scale
    assert lib.moe_combine_nvfp4(None, None, None, 4, 2, 100, None, None, None, None, None) == 1
    assert lib.moe_combine_nvfp4(1 << 20, 1 << 20, None, 4, 2, 128, None, None, None, 1 << 20, None) == 1
    assert lib.moe_fq4_scale_from_amax(None, None, None) == 1
    # batched layout: max_tokens < 1, or more than 2^31 rows
    assert lib.moe_permute_batched(None, 4, 2, 8, 0, 0, None, 128, 0, None, None, None, None, None, None, None, 0,
                                   None, None, 0, None, None, None) == 1
    assert lib.moe_grouped_gemm_batched(None, None, None, 1, 0, 128, 256, None, None, 1, None, None, 0, 0, None,
                                        None, None, None, None) == 1
    assert lib.moe_grouped_gemm_batched(None, None, None, 1025, 1 << 22, 128, 256, None, None, 1025, None, None, 0,
                                        0, None, None, None, None, None) == 1
    # fused down projection + combine: tokens but no row capacity, or K out of range
    assert lib.moe_grouped_gemm_combine(None, None, None, 0, 0, 0, 128, 256, None, None, 1, None, None, 0, None,
                                        None, None, None, None, 4, 2, None, None, None, None, None, None) == 1
    assert lib.moe_grouped_gemm_combine(None, None, None, 1, 0, 16, 128, 256, None, None, 1, None, None, 0, None,
                                        None, None, None, None, 4, 33, None, None, None, None, None, None) == 1


def test_weight_tiles_host_checks(lib):
    """The tile layout's host-side checks (nothing is launched): the layer descriptor flag is
    0 or 1 and does not change the workspace; moe_pack_weights refuses bad sizes, misaligned
    or overlapping buffers and does nothing for an empty tensor; a tiled grouped GEMM whose box
    coordinates would pass 2^31 is refused; SM pairs with tiled weights are refused."""
    d = moe.LayerDesc(128, 7168, 2048, 256, 8, moe.MOE_BF16, 1)
    n0 = lib.moe_layer_workspace_bytes(ctypes.byref(d))
    d.weight_tiles = 1
    assert lib.moe_layer_workspace_bytes(ctypes.byref(d)) == n0 > 0
    d.weight_tiles = 2
    assert lib.moe_layer_workspace_bytes(ctypes.byref(d)) == 0
    a, b = 1 << 30, 1 << 34          # device-looking addresses, never dereferenced
    assert lib.moe_pack_weights(a, 0, 256, 256, moe.MOE_BF16, b, None) == 0
    assert lib.moe_pack_weights(a, 2, 200, 256, moe.MOE_BF16, b, None) == 1       # N % 128
    assert lib.moe_pack_weights(a, 2, 256, 192, moe.MOE_BF16, b, None) == 1       # K % 128
    assert lib.moe_pack_weights(a, 2, 256, 256, 7, b, None) == 1                  # dtype
    assert lib.moe_pack_weights(a + 8, 2, 256, 256, moe.MOE_BF16, b, None) == 1   # alignment
    assert lib.moe_pack_weights(a, 2, 256, 256, moe.MOE_BF16, a + 4096, None) == 1  # overlap
    assert lib.moe_pack_weights(None, 2, 256, 256, moe.MOE_BF16, b, None) == 1
    # 70000 matrices of 4096 x 7168 BF16: 3.2e10 boxes rows, past int32
    big = lib.moe_grouped_gemm(a, None, b, 1, 128, 7168, 4096, a, None, 70000, None, None,
                               moe.MOE_BF16 | moe.MOE_W_TILED, moe.MOE_EPI_NONE, b, None, None, None)
    assert big == 1
    dp = moe.LayerDesc(128, 7168, 2048, 256, 8, moe.MOE_BF16, 0)
    dp.gemm_pairs = 1
    dp.weight_tiles = 1
    n = lib.moe_layer_workspace_bytes(ctypes.byref(dp))
    wts = moe.LayerWeights(a, None, a, None, None, None, None, None)
    code = lib.moe_layer_forward(ctypes.byref(dp), ctypes.byref(wts), None, None, a, a, a, None, None, a, b, n,
                                 None, None)
    assert code == 3
