"""GPU parity of the gate/up projection with fused SwiGLU (nvfp4_gemv_swiglu)
and of the dense SwiGLU FFN (nvfp4_ffn_swiglu) against the CPU oracle.

Tolerance as for the GEMV: |h_gpu - h_ref| <= 1e-2 * (|h_ref| + 1), h_ref the
oracle's unrounded fp64 value.  Inputs: W ~ N(0, 0.02) quantized by the oracle
(gate and up rows interleaved, one tensor), X ~ N(0, 1) bf16 (synth.py).
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


def joint_gate_up(F, K, seed):
    w = np.empty((2 * F, K), dtype=np.float32)
    w[0::2] = synth.weights_f32(F, K, seed)
    w[1::2] = synth.weights_f32(F, K, seed + 1)
    return oracle.quantize(w)


def dev_weights(packed, scale, g):
    return (torch.from_numpy(np.ascontiguousarray(packed)).cuda(), torch.from_numpy(np.ascontiguousarray(scale)).cuda(),
            torch.tensor([g], dtype=torch.float32, device="cuda"))


def dev_x(x16):
    return torch.from_numpy(np.ascontiguousarray(x16).view(np.int16)).cuda().view(torch.bfloat16)


def host_bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def as_f64(b16):
    return torch.from_numpy(np.ascontiguousarray(b16).view(np.int16)).view(torch.bfloat16).double().numpy()


def assert_close(got16, ref64):
    err = np.abs(as_f64(got16) - ref64)
    bad = ~(err <= TOL * (np.abs(ref64) + 1.0))
    assert not bad.any(), f"{bad.sum()} of {bad.size} out of tolerance; worst {err.max()}"


@pytest.mark.parametrize("F,K,n", [(64, 256, 1), (200, 1024, 3), (1024, 2048, 8), (1536, 5120, 16), (4096, 5120, 4)])
def test_gemv_swiglu_matches_oracle(F, K, n):
    packed, scale, g = joint_gate_up(F, K, seed=F + K)
    x = synth.activations_bf16(n, K, seed=7)
    h = nv.nvfp4_gemv_swiglu(*dev_weights(packed, scale, g), dev_x(x))
    torch.cuda.synchronize()
    h64, _ = oracle.gemv_swiglu(packed, scale, g, x)
    assert_close(host_bits(h), h64)
    assert nv.nvfp4_device_error() == 0


def test_gemv_swiglu_batched_equals_single_token_calls():
    F, K, n = 1024, 5120, 8
    packed, scale, g = joint_gate_up(F, K, seed=3)
    x = synth.activations_bf16(n, K, seed=4)
    w = dev_weights(packed, scale, g)
    xt = dev_x(x)
    hb = host_bits(nv.nvfp4_gemv_swiglu(*w, xt))
    for t in range(n):
        ht = host_bits(nv.nvfp4_gemv_swiglu(*w, xt[t:t + 1].contiguous()))
        assert np.array_equal(ht[0], hb[t]), t


@pytest.mark.parametrize("n", [4, 24])  # 24: both projections take the 32-token mode
def test_ffn_swiglu_matches_oracle(n):
    D, F = 1024, 2048
    gu = joint_gate_up(F, D, seed=21)
    down = oracle.quantize(synth.weights_f32(D, F, 23))
    x = synth.activations_bf16(n, D, seed=24)
    h = torch.empty((n, F), dtype=torch.bfloat16, device="cuda")
    y = nv.nvfp4_ffn_swiglu(dev_weights(*gu), dev_weights(*down), dev_x(x), h=h)
    torch.cuda.synchronize()
    h16 = host_bits(h)
    h64, _ = oracle.gemv_swiglu(*gu, x)
    assert_close(h16, h64)
    # the down projection of the GPU's own h, exactly as the GEMV's parity bar
    y64, _ = oracle.gemv(*down, h16)
    assert_close(host_bits(y), y64)
    assert nv.nvfp4_device_error() == 0


@pytest.mark.parametrize("n,variant", [(1, "auto"), (3, "auto"), (4, "auto"), (8, "auto"), (4, "tc"), (24, "tc")])
def test_down_projection_reads_h_written_by_the_kernel_ahead(n, variant):
    """The down projection launches before the gate/up kernel ahead of it has
    finished (programmatic dependent launch) and must read h only as that
    kernel left it: h starts as NaN, so any read of it from before shows."""
    D, F = 1024, 2048
    gu = dev_weights(*joint_gate_up(F, D, seed=21))
    down = dev_weights(*oracle.quantize(synth.weights_f32(D, F, 23)))
    x = dev_x(synth.activations_bf16(n, D, seed=24))
    v = nv.VARIANT_TC if variant == "tc" else nv.VARIANT_AUTO
    h = torch.empty((n, F), dtype=torch.bfloat16, device="cuda")
    nv.nvfp4_gemv_swiglu(*gu, x, h=h)
    torch.cuda.synchronize()
    y_ref = host_bits(nv.nvfp4_gemv_batched_ex(*down, h, variant=v))  # h final before the launch
    for _ in range(3):
        h2 = torch.full((n, F), float("nan"), dtype=torch.bfloat16, device="cuda")
        nv.nvfp4_gemv_swiglu(*gu, x, h=h2)
        y = host_bits(nv.nvfp4_gemv_batched_ex(*down, h2, variant=v))
        assert np.array_equal(host_bits(h2), host_bits(h))
        assert np.array_equal(y, y_ref)
    assert nv.nvfp4_device_error() == 0


def test_gemv_swiglu_needs_the_tcgen05_path():
    packed, scale, g = joint_gate_up(32, 784, seed=5)   # K % 256 != 0
    x = synth.activations_bf16(2, 784, seed=6)
    with pytest.raises(nv.Nvfp4Error) as ei:
        nv.nvfp4_gemv_swiglu(*dev_weights(packed, scale, g), dev_x(x))
    assert ei.value.status == nv.NVFP4_ERR_UNSUPPORTED
