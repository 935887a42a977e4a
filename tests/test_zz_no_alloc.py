"""The allocation-free entry point, nvfp4_gemv_batched_noalloc.

Some callers cannot call cudaMalloc: engines that reserve almost all device
memory in their own pool up front, code that must not allocate once serving
has started (an allocation can synchronize the device), and plugins that only
receive pointers from a host program owning the memory.  For them the library
keeps the kernel's scratch in a static device array.  These tests call that
entry point through the C ABI (ctypes): twice in a row against the ordinary
entry point (same plan, so bit for bit) and sampled points of the oracle
within the parity tolerance; a deep-K call of 32 tokens (two 16-token FP4
passes, as the _ex entry point with an 8 MiB workspace); and a call refused
because no plan fits.  It lives in its own file, collected last, and needs no state
from earlier tests.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import nvfp4_weight_quantized_gemv_gb300 as nv
import oracle
import synth

pytestmark = pytest.mark.gpu
TOL = 1e-2


def _bf16_to_f64(t):
    return t.double().cpu().numpy()


def _case(N, K, n, wseed, xseed):
    packed, scale, g = oracle.quantize(synth.weights_f32(N, K, wseed))
    x = synth.activations_bf16(n, K, xseed)
    wp = torch.from_numpy(packed).cuda()
    ws = torch.from_numpy(scale).cuda()
    gs = torch.tensor([g], dtype=torch.float32, device="cuda")
    xt = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    return wp, ws, gs, xt


@pytest.mark.parametrize("N,K,n", [(14336, 5120, 4), (700, 1280, 3), (14336, 5120, 32)])
def test_noalloc_matches_default_entry_point_twice(N, K, n):
    """Same plan as the default entry point, so the same bits; both within the
    parity tolerance of the oracle."""
    nv.build()
    oracle.build()
    L = nv.lib()
    stream = torch.cuda.current_stream()
    for call in range(2):
        wp, ws, gs, xt = _case(N, K, n, 10 + call, 20 + call)
        y_ref = torch.empty((n, N), dtype=torch.bfloat16, device="cuda")
        y_new = torch.full((n, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        st = L.nvfp4_gemv_batched(wp.data_ptr(), ws.data_ptr(), gs.data_ptr(), xt.data_ptr(), y_ref.data_ptr(),
                                  n, N, K, ctypes.c_void_p(stream.cuda_stream))
        assert st == nv.NVFP4_OK, nv.nvfp4_last_error()
        st = L.nvfp4_gemv_batched_noalloc(wp.data_ptr(), ws.data_ptr(), gs.data_ptr(), xt.data_ptr(),
                                          y_new.data_ptr(), n, N, K, ctypes.c_void_p(stream.cuda_stream))
        assert st == nv.NVFP4_OK, nv.nvfp4_last_error()
        torch.cuda.synchronize()
        assert torch.equal(y_new.view(torch.int16), y_ref.view(torch.int16)), f"call {call}"
        _check_sampled(wp, ws, gs, xt, y_new, call)
    assert nv.nvfp4_device_error() == 0


def _check_sampled(wp, ws, gs, xt, y, seed):
    n, N = y.shape
    packed, scale = wp.cpu().numpy(), ws.cpu().numpy()
    x = xt.view(torch.int16).cpu().numpy().view(np.uint16)
    rng = np.random.Generator(np.random.PCG64(seed))
    rows = np.concatenate([[0, N - 1], rng.integers(0, N, 200)])
    toks = rng.integers(0, n, rows.shape[0])
    ref, _ = oracle.gemv_points(packed, scale, float(gs.item()), x, toks, rows)
    got = _bf16_to_f64(y)[toks, rows]
    assert np.all(np.abs(got - ref) <= TOL * (np.abs(ref) + 1.0))


def test_noalloc_two_passes_at_deep_k():
    """n = 32 at K = 16384: AUTO's plan is two 16-token FP4 passes, within the
    8 MiB static scratch -- the plan, and the bits, of the _ex entry point
    given an 8 MiB workspace."""
    nv.build()
    oracle.build()
    N, K, n = 14336, 16384, 32
    cap = 8 << 20
    assert nv.nvfp4_gemv_workspace_size(n, N, K) <= cap
    plan = nv.nvfp4_gemv_plan(n, N, K, workspace_bytes=cap)
    assert plan["tile_tokens"] == [16, 16] and plan["variant"] == "fp4"
    wp, ws, gs, xt = _case(N, K, n, 40, 41)
    work = torch.zeros(cap, dtype=torch.uint8, device="cuda")
    y_ex = nv.nvfp4_gemv_batched_ex(wp, ws, gs, xt, workspace=work)
    L = nv.lib()
    stream = torch.cuda.current_stream()
    y_new = torch.full((n, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = L.nvfp4_gemv_batched_noalloc(wp.data_ptr(), ws.data_ptr(), gs.data_ptr(), xt.data_ptr(),
                                      y_new.data_ptr(), n, N, K, ctypes.c_void_p(stream.cuda_stream))
    assert st == nv.NVFP4_OK, nv.nvfp4_last_error()
    torch.cuda.synchronize()
    assert torch.equal(y_new.view(torch.int16), y_ex.view(torch.int16))
    _check_sampled(wp, ws, gs, xt, y_new, 42)
    assert nv.nvfp4_device_error() == 0


def test_noalloc_refuses_a_plan_beyond_the_static_scratch():
    """17 tokens over 262144 rows of K = 33024 (beyond the FP4 kernel's K): even
    the tcgen05 kernel's 8-token passes need far more than 8 MiB of split-tile
    scratch; the call is refused before anything is enqueued."""
    nv.build()
    N, K, n = 262144, 33024, 17
    assert nv.nvfp4_gemv_workspace_size(8, N, K) > (8 << 20)
    L = nv.lib()
    p = ctypes.c_void_p(1 << 20)      # aligned, never dereferenced: the refusal comes first
    assert L.nvfp4_gemv_batched_noalloc(p, p, p, p, p, n, N, K, None) == nv.NVFP4_ERR_WORKSPACE
    assert "static scratch" in nv.nvfp4_last_error()


def test_noalloc_rejects_bad_arguments():
    nv.build()
    L = nv.lib()
    p = ctypes.c_void_p(256)
    assert L.nvfp4_gemv_batched_noalloc(p, p, p, p, p, 1, 128, 24, None) == nv.NVFP4_ERR_INVALID_ARG
    assert L.nvfp4_gemv_batched_noalloc(None, p, p, p, p, 1, 128, 256, None) == nv.NVFP4_ERR_INVALID_ARG
