"""The allocation-free entry point, nvfp4_gemv_batched_noalloc.

Some callers cannot call cudaMalloc: engines that reserve almost all device
memory in their own pool up front, code that must not allocate once serving
has started (an allocation can synchronize the device), and plugins that only
receive pointers from a host program owning the memory.  For them the library
keeps the kernel's scratch in a static device array.  This test calls that
entry point through the C ABI (ctypes) twice in a row and checks each result
against the ordinary entry point's, within the parity tolerance used by the
other GPU tests.  It lives in its own file, collected last, and needs no state
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


@pytest.mark.parametrize("N,K,n", [(14336, 5120, 4), (700, 1280, 3)])
def test_noalloc_matches_default_entry_point_twice(N, K, n):
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
        ref, new = _bf16_to_f64(y_ref), _bf16_to_f64(y_new)
        assert not np.isnan(new).any()
        assert np.all(np.abs(new - ref) <= TOL * (np.abs(ref) + 1.0)), f"call {call}"
    assert nv.nvfp4_device_error() == 0


def test_noalloc_rejects_bad_arguments():
    nv.build()
    L = nv.lib()
    p = ctypes.c_void_p(256)
    assert L.nvfp4_gemv_batched_noalloc(p, p, p, p, p, 1, 128, 24, None) == nv.NVFP4_ERR_INVALID_ARG
    assert L.nvfp4_gemv_batched_noalloc(None, p, p, p, p, 1, 128, 256, None) == nv.NVFP4_ERR_INVALID_ARG
