"""The kernels' failure path on the GPU, without a fault: a wait that nothing
ends gives up after the wait limit, the host reads NVFP4_ERR_DEVICE_TIMEOUT
from the device error word, and the context stays usable (a GEMV right after
still matches the oracle)."""
from __future__ import annotations

import time

import numpy as np
import pytest
import torch

import nvfp4_weight_quantized_gemv_gb300 as nv
import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    nv.build()
    oracle.build()


def test_bounded_wait_times_out_and_the_context_survives():
    assert nv.nvfp4_device_error() == 0
    t0 = time.monotonic()
    nv.nvfp4_selftest_wait_timeout()
    with pytest.raises(nv.Nvfp4Error) as ei:
        nv.nvfp4_device_error()  # synchronizes: the kernel has given up by now
    assert ei.value.status == nv.NVFP4_ERR_DEVICE_TIMEOUT
    assert 1.5 < time.monotonic() - t0 < 30.0  # the 2 s limit, give or take the launch
    assert nv.nvfp4_device_error() == 0  # read and cleared

    N, K, n = 512, 1024, 5
    packed, scale, g = oracle.quantize(synth.weights_f32(N, K, 0))
    x = synth.activations_bf16(n, K, 1)
    y64, _ = oracle.gemv(packed, scale, g, x)
    wp = torch.from_numpy(packed).cuda()
    ws = torch.from_numpy(scale).cuda()
    gs = torch.tensor([g], dtype=torch.float32, device="cuda")
    xt = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    y = nv.nvfp4_gemv_batched(wp, ws, gs, xt)
    torch.cuda.synchronize()
    yv = y.double().cpu().numpy()
    assert np.all(np.abs(yv - y64) <= 1e-2 * (np.abs(y64) + 1.0))
    assert nv.nvfp4_device_error() == 0
