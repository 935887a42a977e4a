"""GPU parity of the mid-M widths (n = 17..64 tokens, the widths atlas #266
serves with its mid-M tile GEMM: verify and prefill batches): AUTO's FP4
kernel in passes of 16 tokens (the weights of a pass that another follows
kept in L2), and the tcgen05 kernel's 32-token mode (X converted once to f16
x 2^-8 and streamed per unit through a ring, 32 tokens per read of W).

Tolerance as for the GEMV: |y_gpu - y_ref| <= 1e-2 * (|y_ref| + 1), y_ref the
oracle's unrounded fp64 value.  Each kernel's partition does not depend on n,
so a batched call equals the single-token calls of the same kernel bit for bit
(atlas #266, "Correctness argument").  Inputs: oracle-quantized W ~ N(0, 0.02),
X ~ N(0, 1) bf16 (synth.py).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import nvfp4_weight_quantized_gemv_gb300 as nv
import oracle
import synth

pytestmark = pytest.mark.gpu
TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def built():
    nv.build()
    oracle.build()


def make_case(N, K, n, wseed=0, xseed=1, outlier=0.0):
    w = synth.weights_f32(N, K, wseed)
    packed, scale, g = oracle.quantize(w)
    x = synth.activations_bf16(n, K, xseed, outlier)
    return packed, scale, g, x


def to_gpu(packed, scale, g, x):
    wp = torch.from_numpy(np.ascontiguousarray(packed)).cuda()
    ws = torch.from_numpy(np.ascontiguousarray(scale)).cuda()
    gs = torch.tensor([g], dtype=torch.float32, device="cuda")
    xt = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda().view(torch.bfloat16)
    return wp, ws, gs, xt


def bits(t):
    torch.cuda.synchronize()
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def as_f64(y16):
    return torch.from_numpy(np.ascontiguousarray(y16).view(np.int16)).view(torch.bfloat16).double().numpy()


def assert_close(y16, y64):
    err = np.abs(as_f64(y16) - y64)
    bad = ~(err <= TOL * (np.abs(y64) + 1.0))
    assert not bad.any(), f"{bad.sum()} of {bad.size} out of tolerance; worst {err.max()}"


@pytest.mark.parametrize("variant", ["auto", "tc"])
@pytest.mark.parametrize("N,K,n,tiles,tc_tiles", [
    (1000, 1024, 17, [16, 1], [17]),          # a one-token second pass / one 32-token pass
    (384, 2048, 32, [16, 16], [32]),          # two full FP4 passes / a full 32-token pass
    (2000, 512, 24, [16, 8], [24]),           # short segments (two units per row block)
    (256, 8192, 20, [16, 4], [20]),           # deep K
    (700, 1280, 40, [16, 16, 8], [32, 8]),    # three passes / a second pass of 8 tokens
    (300, 768, 64, [16, 16, 16, 16], [32, 32]),
    (129, 256, 33, [16, 16, 1], [32, 1]),     # one unit per row block, a one-token tail pass
])
def test_mid_m_full_output(variant, N, K, n, tiles, tc_tiles):
    v = nv.VARIANT_TC if variant == "tc" else 0
    assert nv.nvfp4_gemv_plan(n, N, K, variant=v)["tile_tokens"] == (tc_tiles if variant == "tc" else tiles)
    packed, scale, g, x = make_case(N, K, n, 3, 4, outlier=0.01)
    y64, _ = oracle.gemv(packed, scale, g, x)
    wp, ws, gs, xt = to_gpu(packed, scale, g, x)
    assert_close(bits(nv.nvfp4_gemv_batched_ex(wp, ws, gs, xt, variant=v)), y64)


@pytest.mark.parametrize("n", [32, 40])
def test_mid_m_equals_single_token_calls(n):
    N, K = 1536, 2048
    packed, scale, g, x = make_case(N, K, n, 5, 6)
    wp, ws, gs, xt = to_gpu(packed, scale, g, x)
    for v in (0, nv.VARIANT_TC):  # AUTO (FP4 passes) and the tcgen05 32-token mode
        full = bits(nv.nvfp4_gemv_batched_ex(wp, ws, gs, xt, variant=v))
        for t in range(n):
            one = bits(nv.nvfp4_gemv_batched_ex(wp, ws, gs, xt[t:t + 1].contiguous(), variant=v))
            assert np.array_equal(one[0], full[t]), (v, t)


@pytest.mark.parametrize("n", [32, 64])
def test_mid_m_full_size_qkv_sampled(n):
    N, K = 14336, 5120
    packed, scale, g, x = make_case(N, K, n, 0, 1)
    wp, ws, gs, xt = to_gpu(packed, scale, g, x)
    y16 = bits(nv.nvfp4_gemv_batched(wp, ws, gs, xt))
    assert not np.isnan(as_f64(y16)).any()
    rng = np.random.Generator(np.random.PCG64(40 + n))
    rows = np.concatenate([[0, 1, 127, 128, N - 129, N - 128, N - 1], rng.integers(0, N, 400)])
    toks = rng.integers(0, n, rows.shape[0])
    ref64, _ = oracle.gemv_points(packed, scale, g, x, toks, rows)
    assert_close(y16[toks, rows], ref64)
    for t in (0, 17, n - 1):  # batched == single token on the full-size launch configuration
        one = bits(nv.nvfp4_gemv_batched(wp, ws, gs, xt[t:t + 1].contiguous()))
        assert np.array_equal(one[0], y16[t]), t


def test_mid_m_activation_beyond_f16_range_is_rescaled():
    N, K, n = 256, 1024, 20
    packed, scale, g, _ = make_case(N, K, 1, 1, 1)
    xf = synth.activations_f32(n, K, 1)
    xf[1, 17] = 3.0e5             # beyond f16's range, inside the 2^-8 prescale's
    xf[19, 900] = -1.0e6
    x = synth.to_bf16_bits(xf)
    y64, _ = oracle.gemv(packed, scale, g, x)
    wp, ws, gs, xt = to_gpu(packed, scale, g, x)
    assert_close(bits(nv.nvfp4_gemv_batched(wp, ws, gs, xt)), y64)
    assert nv.nvfp4_device_error() == 0


def test_mid_m_swiglu():
    F, K, n = 1024, 2048, 24
    w = np.empty((2 * F, K), dtype=np.float32)
    w[0::2] = synth.weights_f32(F, K, 7)
    w[1::2] = synth.weights_f32(F, K, 8)
    packed, scale, g = oracle.quantize(w)
    x = synth.activations_bf16(n, K, 9)
    h64, _ = oracle.gemv_swiglu(packed, scale, g, x)
    wp, ws, gs, xt = to_gpu(packed, scale, g, x)
    assert_close(bits(nv.nvfp4_gemv_swiglu(wp, ws, gs, xt)), h64)


def test_mid_m_caller_workspace_and_fallback():
    N, K, n = 2048, 2048, 32
    packed, scale, g, x = make_case(N, K, n, 2, 3)
    y64, _ = oracle.gemv(packed, scale, g, x)
    wp, ws, gs, xt = to_gpu(packed, scale, g, x)
    big = torch.zeros(nv.nvfp4_gemv_workspace_size(n, N, K), dtype=torch.uint8, device="cuda")
    y_big = bits(nv.nvfp4_gemv_batched_ex(wp, ws, gs, xt, workspace=big))
    assert_close(y_big, y64)
    # a scratch too small for the FP4 plan but enough for the tcgen05 kernel's
    # 8-token passes: the call takes those (another kernel: within the tolerance)
    small_bytes = nv.nvfp4_gemv_workspace_size(8, N, K, variant=nv.VARIANT_TC)
    assert small_bytes < big.numel()
    plan = nv.nvfp4_gemv_plan(n, N, K, workspace_bytes=small_bytes)
    assert plan["variant"] == "tc" and plan["tile_tokens"] == [8, 8, 8, 8]
    small = torch.zeros(small_bytes, dtype=torch.uint8, device="cuda")
    assert_close(bits(nv.nvfp4_gemv_batched_ex(wp, ws, gs, xt, workspace=small)), y64)
    y = torch.empty((n, N), dtype=torch.bfloat16, device="cuda")
    nv.nvfp4_gemv_batched_noalloc(wp, ws, gs, xt, y)
    assert np.array_equal(bits(y), y_big)


@pytest.mark.parametrize("num_ctas,stages", [(1, 2), (7, 4), (150, 8), (0, 2)])
def test_mid_m_grid_and_ring_options(num_ctas, stages):
    N, K, n = 700, 1280, 24
    packed, scale, g, x = make_case(N, K, n, 7, 8)
    y64, _ = oracle.gemv(packed, scale, g, x)
    wp, ws, gs, xt = to_gpu(packed, scale, g, x)
    y = nv.nvfp4_gemv_batched_ex(wp, ws, gs, xt, variant=nv.VARIANT_TC, num_ctas=num_ctas, stages=stages)
    assert_close(bits(y), y64)


def test_no_device_error_recorded():
    assert nv.nvfp4_device_error() == 0
