"""Host-side tests of the C-ABI library: no GPU needed.

  - the library loads and exports every function include/nvfp4_gemv.h declares;
  - argument validation returns the documented status without touching a GPU;
  - the tile policy (greedy 3/2/1 as on the pages, one pass otherwise);
  - the product's host quantizer (nvfp4_quantize_ref) equals the oracle's
    quantizer byte for byte (integer codes decided in fp32 on both sides).
"""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np
import pytest

import nvfp4_weight_quantized_gemv_gb300 as nv
import oracle
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    nv.build()
    oracle.build()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "nvfp4_gemv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nvfp4_\w+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    names = declared_functions()
    assert "nvfp4_gemv_batched" in names and "nvfp4_quantize_ref" in names
    L = ctypes.CDLL(nv.LIB_PATH)
    for name in names:
        assert hasattr(L, name), name
    assert set(names) == set(nv.EXPORTS)
    assert nv.nvfp4_version() >= 100


def test_debug_bounds_build_exports_the_same_symbols():
    from nvfp4_weight_quantized_gemv_gb300 import buildlib
    path = buildlib.build(debug_bounds=True)
    assert path == nv.DEBUG_LIB_PATH
    L = ctypes.CDLL(path)
    for name in declared_functions():
        assert hasattr(L, name), name


def test_validation_errors_without_gpu():
    L = nv.lib()
    p = ctypes.c_void_p(16)
    # n < 0, N < 1, K not a multiple of 16, null pointers
    assert L.nvfp4_gemv_batched(p, p, p, p, p, -1, 128, 256, None) == nv.NVFP4_ERR_INVALID_ARG
    assert "n = -1" in nv.nvfp4_last_error()
    assert L.nvfp4_gemv_batched(p, p, p, p, p, 1, 0, 256, None) == nv.NVFP4_ERR_INVALID_ARG
    assert L.nvfp4_gemv_batched(p, p, p, p, p, 1, 128, 24, None) == nv.NVFP4_ERR_INVALID_ARG
    assert L.nvfp4_gemv_batched(p, p, p, p, p, 1, 128, 8, None) == nv.NVFP4_ERR_INVALID_ARG
    assert L.nvfp4_gemv_batched(None, p, p, p, p, 1, 128, 256, None) == nv.NVFP4_ERR_INVALID_ARG
    assert L.nvfp4_gemv_batched(p, p, p, p, None, 1, 128, 256, None) == nv.NVFP4_ERR_INVALID_ARG
    # n == 0 is a no-op even with null pointers
    assert L.nvfp4_gemv_batched(None, None, None, None, None, 0, 128, 256, None) == nv.NVFP4_OK
    o = nv._opts(variant=7)
    assert L.nvfp4_gemv_batched_ex(p, p, p, p, p, 1, 128, 256, None, ctypes.byref(o)) == nv.NVFP4_ERR_INVALID_ARG
    # the tcgen05 kernel takes an even number of weight stages
    with pytest.raises(nv.Nvfp4Error, match="even"):
        nv.nvfp4_gemv_plan(3, 4096, 4096, variant=nv.VARIANT_TC, stages=5)
    assert nv.nvfp4_gemv_plan(3, 4096, 4096, variant=nv.VARIANT_MMA, stages=5)["stages"] == 5
    w = np.zeros((2, 24), dtype=np.float32)
    with pytest.raises(nv.Nvfp4Error):
        nv.nvfp4_quantize_ref(w)


def test_grouped_expert_validation_without_gpu():
    L = nv.lib()
    a = ctypes.c_void_p(4096)
    f = L.nvfp4_moe_gemv_grouped
    assert f(None, a, a, a, a, a, a, 4, 8, 2, 64, 256, 0, None) == nv.NVFP4_ERR_INVALID_ARG
    assert f(a, a, a, a, a, a, a, 0, 8, 2, 64, 256, 0, None) == nv.NVFP4_ERR_INVALID_ARG      # E
    assert f(a, a, a, a, a, a, a, 1025, 8, 2, 64, 256, 0, None) == nv.NVFP4_ERR_INVALID_ARG   # E > 1024
    assert f(a, a, a, a, a, a, a, 4, 8, 2, 64, 240, 0, None) == nv.NVFP4_ERR_INVALID_ARG      # K % 32
    assert f(a, a, a, a, a, a, a, 4, 8, 2, 64, 8192, 0, None) == nv.NVFP4_ERR_INVALID_ARG     # K too large
    assert f(a, a, a, a, a, a, a, 4, 8, 2, 72, 256, 1, None) == nv.NVFP4_ERR_INVALID_ARG      # N % 16
    assert f(a, a, a, a, a, a, a, 4, 8, 2, 64, 256, 2, None) == nv.NVFP4_ERR_INVALID_ARG      # swiglu flag
    b = ctypes.c_void_p(4096 + 8)
    assert f(b, a, a, a, a, a, a, 4, 8, 2, 64, 256, 0, None) == nv.NVFP4_ERR_MISALIGNED
    assert f(a, a, a, a, a, a, a, 4, 0, 2, 64, 256, 0, None) == nv.NVFP4_OK                  # no assignment


def test_device_quantizer_validation_without_gpu():
    """nvfp4_quantize / nvfp4_quantize_bf16 reject bad arguments before any CUDA call."""
    L = nv.lib()
    a16, a8, a4 = ctypes.c_void_p(4096), ctypes.c_void_p(4096 + 8), ctypes.c_void_p(4096 + 4)
    for fn in (L.nvfp4_quantize, L.nvfp4_quantize_bf16):
        assert fn(None, 4, 64, a16, a16, a16, None) == nv.NVFP4_ERR_INVALID_ARG
        assert fn(a16, 4, 64, a16, None, a16, None) == nv.NVFP4_ERR_INVALID_ARG
        assert fn(a16, 0, 64, a16, a16, a16, None) == nv.NVFP4_ERR_INVALID_ARG
        assert fn(a16, 4, 24, a16, a16, a16, None) == nv.NVFP4_ERR_INVALID_ARG
        assert "multiple of 16" in nv.nvfp4_last_error()
        assert fn(a16, 4, 0, a16, a16, a16, None) == nv.NVFP4_ERR_INVALID_ARG
        assert fn(a16, 1 << 30, 1 << 14, a16, a16, a16, None) == nv.NVFP4_ERR_INVALID_ARG
        assert fn(a8, 4, 64, a16, a16, a16, None) == nv.NVFP4_ERR_MISALIGNED      # weights need 16 B
        assert fn(a16, 4, 64, a4, a16, a16, None) == nv.NVFP4_ERR_MISALIGNED      # codes need 8 B
        assert fn(a16, 4, 64, a8, a16, ctypes.c_void_p(4098), None) == nv.NVFP4_ERR_MISALIGNED


def test_greedy_321_tiling_matches_the_pages():
    # atlas #266 "What it does": greedy 3s then a 2-or-1 remainder; n = 8 -> 3 weight reads
    expect = {1: [1], 2: [2], 3: [3], 4: [3, 1], 5: [3, 2], 8: [3, 3, 2], 16: [3, 3, 3, 3, 3, 1]}
    for n, tiles in expect.items():
        plan = nv.nvfp4_gemv_plan(n, 14336, 5120, tiling=nv.TILING_GREEDY_321)
        assert plan["tile_tokens"] == tiles and plan["passes"] == len(tiles)
    assert nv.nvfp4_gemv_plan(8, 14336, 5120, tiling=nv.TILING_GREEDY_321)["passes"] == 3


def test_one_pass_plan():
    for n in (1, 4, 8, 16):
        plan = nv.nvfp4_gemv_plan(n, 14336, 5120)
        assert plan["variant"] == "fp4" and plan["tiling"] == "one_pass"
        assert plan["passes"] == 1 and plan["tile_tokens"] == [n]
        assert plan["units"] == (14336 // 128) * (5120 // 256)
        assert 4 <= plan["stages"] <= 16 and plan["smem_bytes"] <= 232448 - 4096
        tc = nv.nvfp4_gemv_plan(n, 14336, 5120, variant=nv.VARIANT_TC)
        assert tc["units"] == (14336 // 128) * (5120 // 256)
        assert 2 <= tc["stages"] <= 8 and tc["stages"] % 2 == 0 and tc["smem_bytes"] <= 232448
        mma = nv.nvfp4_gemv_plan(n, 14336, 5120, variant=nv.VARIANT_MMA)
        assert mma["units"] == (14336 // 128) * (5120 // 128)
    # the FP4 kernel takes K up to 32768; beyond, AUTO takes the tcgen05 kernel
    assert nv.nvfp4_gemv_plan(4, 256, 32768)["variant"] == "fp4"
    assert nv.nvfp4_gemv_plan(4, 256, 32768 + 256)["variant"] == "tc"
    with pytest.raises(nv.Nvfp4Error):
        nv.nvfp4_gemv_plan(4, 256, 32768 + 256, variant=nv.VARIANT_FP4)
    # greedy 3/2/1 tiling on the FP4 kernel: tiles of 3 tokens
    assert nv.nvfp4_gemv_plan(8, 14336, 5120, tiling=nv.TILING_GREEDY_321)["tile_tokens"] == [3, 3, 2]
    assert nv.nvfp4_gemv_plan(8, 14336, 5120, tiling=nv.TILING_GREEDY_321)["variant"] == "fp4"
    # a declared scratch size too small for the FP4 plan: the tcgen05 kernel
    f4 = nv.nvfp4_gemv_workspace_size(8, 14336, 5120)
    tc8 = nv.nvfp4_gemv_workspace_size(8, 14336, 5120, variant=nv.VARIANT_TC)
    if tc8 < f4:
        assert nv.nvfp4_gemv_plan(8, 14336, 5120, workspace_bytes=tc8)["variant"] == "tc"
    assert nv.nvfp4_gemv_plan(8, 14336, 5120, workspace_bytes=f4)["variant"] == "fp4"
    # more than 16 tokens: FP4 passes of 16 (the tcgen05 kernel's 32-token mode on request)
    assert nv.nvfp4_gemv_plan(20, 4096, 4096)["tile_tokens"] == [16, 4]
    assert nv.nvfp4_gemv_plan(40, 14336, 5120)["tile_tokens"] == [16, 16, 8]
    assert nv.nvfp4_gemv_plan(40, 14336, 5120)["variant"] == "fp4"
    assert nv.nvfp4_gemv_plan(32, 14336, 5120, variant=nv.VARIANT_TC)["tile_tokens"] == [32]
    assert nv.nvfp4_gemv_plan(64, 14336, 5120, variant=nv.VARIANT_TC)["tile_tokens"] == [32, 32]
    assert nv.nvfp4_gemv_plan(40, 14336, 5120, variant=nv.VARIANT_TC)["tile_tokens"] == [32, 8]
    # an explicit tcgen05 call with a scratch size too small for its 32-token pass: 8-token passes
    tc8s = nv.nvfp4_gemv_workspace_size(8, 14336, 5120, variant=nv.VARIANT_TC)
    assert nv.nvfp4_gemv_workspace_size(32, 14336, 5120, variant=nv.VARIANT_TC) > tc8s
    assert nv.nvfp4_gemv_plan(20, 14336, 5120, variant=nv.VARIANT_TC,
                              workspace_bytes=tc8s)["tile_tokens"] == [8, 8, 4]
    # beyond the FP4 kernel's K: the tcgen05 kernel's 8-token passes
    tc8 = nv.nvfp4_gemv_workspace_size(8, 1024, 33024)
    assert nv.nvfp4_gemv_plan(20, 1024, 33024, workspace_bytes=tc8)["tile_tokens"] == [8, 8, 4]
    # the tcgen05 kernel stages 8 or 32 tokens (9 to 16 take the 32-token mode)
    assert nv.nvfp4_gemv_plan(12, 1024, 8192, variant=nv.VARIANT_TC)["tile_tokens"] == [12]
    # K too large for 16 tokens of X in shared memory: smaller chunks
    p = nv.nvfp4_gemv_plan(16, 1024, 8192)
    assert p["tile_tokens"] == [16]        # FP4: X codes streamed per unit when not resident
    p = nv.nvfp4_gemv_plan(16, 1024, 8192, variant=nv.VARIANT_TC)
    assert p["tile_tokens"] == [16]        # tcgen05: X is streamed per unit, any K fits
    p = nv.nvfp4_gemv_plan(16, 1024, 8192, variant=nv.VARIANT_MMA)
    assert sum(p["tile_tokens"]) == 16 and max(p["tile_tokens"]) < 16
    # K % 256 != 0 -> generic kernel, no workspace
    assert nv.nvfp4_gemv_plan(3, 100, 784)["variant"] == "generic"
    assert nv.nvfp4_gemv_workspace_size(3, 100, 784) == 0
    assert nv.nvfp4_gemv_workspace_size(3, 14336, 5120) > 0
    # the grid never exceeds the number of units
    assert nv.nvfp4_gemv_plan(3, 256, 512)["num_ctas"] == 2 * 2          # FP4: 128 x 256 units
    assert nv.nvfp4_gemv_plan(3, 256, 512, variant=nv.VARIANT_TC)["num_ctas"] == 2 * 2
    assert nv.nvfp4_gemv_plan(3, 256, 512, variant=nv.VARIANT_MMA)["num_ctas"] == 2 * 4


def test_host_quantizer_matches_oracle_bytes():
    for (N, K, seed) in [(64, 512, 0), (37, 272, 1), (5, 16, 2)]:
        w = synth.weights_f32(N, K, seed)
        w[1, :16] *= 1e-5        # subnormal block scale
        w[2, 16:32] = 0.0        # zero block
        p1, s1, g1 = nv.nvfp4_quantize_ref(w)
        p2, s2, g2 = oracle.quantize(w)
        assert g1 == g2
        assert np.array_equal(s1, s2)
        assert np.array_equal(p1, p2)


def test_host_quantizer_golden_case():
    from fractions import Fraction
    from golden_io import fractions, hex_bytes, read_cases
    for case in read_cases("quantize_hand_cases.txt"):
        N, K = int(case["N"][0]), int(case["K"][0])
        w = np.array([float(f) for f in fractions(case["w"])], dtype=np.float32).reshape(N, K)
        packed, scale, g = nv.nvfp4_quantize_ref(w)
        assert Fraction(g) == Fraction(case["g"][0])
        assert scale.ravel().tolist() == hex_bytes(case["scale"])
        assert packed.ravel().tolist() == hex_bytes(case["packed"])
