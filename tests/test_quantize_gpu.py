"""GPU parity of the device NVFP4 quantizer (nvfp4_quantize, nvfp4_quantize_bf16).

The quantizer's outputs are integers (E2M1 codes, E4M3 scales) and one fp32
global scale, decided in fp32 on both sides, so the bar is bit-exact: every
byte and the bits of g equal the oracle's (oracle.quantize) on the same
weights.  bf16 weights are widened exactly to fp32 before the oracle sees them.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import nvfp4_weight_quantized_gemv_gb300 as nv
import oracle
import synth
from golden_io import fractions, hex_bytes, read_cases

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    nv.build()
    oracle.build()


def gpu_quantize(w):
    """w: numpy fp32 array, or numpy uint16 bf16 bit patterns."""
    if w.dtype == np.uint16:
        wt = torch.from_numpy(np.ascontiguousarray(w).view(np.int16)).cuda().view(torch.bfloat16)
    else:
        wt = torch.from_numpy(np.ascontiguousarray(w, dtype=np.float32)).cuda()
    packed, scale, g = nv.nvfp4_quantize(wt)
    torch.cuda.synchronize()
    return packed.cpu().numpy(), scale.cpu().numpy(), g.cpu().numpy()


def bf16_bits_to_f32(b):
    return (np.ascontiguousarray(b).astype(np.uint32) << 16).view(np.float32)


def assert_same(w32, got):
    packed, scale, g = oracle.quantize(w32)
    gp, gs, gg = got
    assert gg.view(np.uint32)[0] == np.float32(g).view(np.uint32), (gg[0], g)
    bad_s = np.argwhere(gs != scale)
    assert bad_s.size == 0, f"{len(bad_s)} scales differ, first at {bad_s[0]}"
    bad_p = np.argwhere(gp != packed)
    assert bad_p.size == 0, f"{len(bad_p)} code bytes differ, first at {bad_p[0]}"


@pytest.mark.parametrize("case", read_cases("quantize_hand_cases.txt"), ids=lambda c: c["name"])
def test_hand_derived_cases(case):
    N, K = int(case["N"][0]), int(case["K"][0])
    w = np.array([float(f) for f in fractions(case["w"])], dtype=np.float32).reshape(N, K)
    gp, gs, gg = gpu_quantize(w)
    assert float(gg[0]) == float(fractions(case["g"])[0])
    assert gs.ravel().tolist() == hex_bytes(case["scale"])
    assert gp.ravel().tolist() == hex_bytes(case["packed"])
    assert nv.nvfp4_device_error() == 0


@pytest.mark.parametrize("N,K", [(1, 16), (3, 48), (37, 368), (128, 5120), (301, 2064)])
def test_random_fp32(N, K):
    w = synth.weights_f32(N, K, seed=N * 7 + K)
    assert_same(w, gpu_quantize(w))


@pytest.mark.parametrize("N,K", [(1, 16), (37, 368), (257, 4096)])
def test_random_bf16(N, K):
    wb = synth.to_bf16_bits(synth.weights_f32(N, K, seed=N + K))
    assert_same(bf16_bits_to_f32(wb), gpu_quantize(wb))


def edge_matrix():
    """g = 1 exactly (amax = 2688), blocks built on exact E2M1 midpoints,
    zero and negative-zero blocks, subnormal E4M3 scales, scales that round to
    zero, and ordinary blocks, over a ragged number of 16-blocks."""
    N, K = 13, 16 * 9
    w = synth.weights_f32(N, K, seed=5, std=3.0)
    w[0, 0] = 2688.0                               # amax -> g = 1, s = 448 there
    mids = np.array([0, .25, .5, .75, 1, 1.25, 1.5, 1.75, 2, 2.5, 3, 3.5, 4, 5, 6, -6], np.float32)
    for r, s in enumerate([448.0, 224.0, 2.0 ** -6, 2.0 ** -7, 3 * 2.0 ** -9, 2.0 ** -9]):
        w[1 + r, 16:32] = mids * np.float32(s)     # bmax = 6 s: exact scale, ties everywhere
        w[1 + r, 32:48] = -mids * np.float32(s)
    w[7, :] = 0.0
    w[8, 0:16] = -0.0
    w[8, 16:32] = np.float32(1e-30)                # s rounds to 0: all codes 0
    w[9, 48:64] = np.float32(2.0 ** -9) * np.arange(16, dtype=np.float32)
    w[10, :] *= np.float32(1e-3)
    w[11, 0:16] = np.float32(6 * 447.9)            # scale just under the saturation point
    w[12, 0:16] = np.float32(6 * 464.0 / 2)        # scale on an E4M3 tie (232)
    return w


def test_edge_cases_fp32():
    w = edge_matrix()
    assert_same(w, gpu_quantize(w))


def test_edge_cases_bf16():
    wb = synth.to_bf16_bits(edge_matrix())
    assert_same(bf16_bits_to_f32(wb), gpu_quantize(wb))


@pytest.mark.parametrize("amax", [0.0, 1e-40, 1e-30, 3.0e38])
def test_extreme_global_scales(amax):
    N, K = 9, 80
    w = synth.weights_f32(N, K, seed=11, std=1.0)
    if amax == 0.0:
        w[:] = 0.0                                 # g = 1, every scale and code 0
    else:
        w = (w / np.abs(w).max() * np.float32(amax)).astype(np.float32)
    assert_same(w, gpu_quantize(w))


def test_full_size_attention_qkv_bf16():
    """The attention qkv projection's shape (N = 14336, K = 5120), bf16 weights."""
    N, K = 14336, 5120
    wb = synth.to_bf16_bits(synth.weights_f32(N, K, seed=3))
    assert_same(bf16_bits_to_f32(wb), gpu_quantize(wb))
    assert nv.nvfp4_device_error() == 0


def test_non_finite_weight_sets_the_error_word():
    w = synth.weights_f32(4, 64, seed=2)
    w[2, 17] = np.inf
    gpu_quantize(w)
    assert nv.nvfp4_device_error() & 16
    assert nv.nvfp4_device_error() == 0            # read clears it
    wb = synth.to_bf16_bits(synth.weights_f32(4, 64, seed=2))
    wb[1, 3] = 0x7FC0                              # bf16 NaN
    gpu_quantize(wb)
    assert nv.nvfp4_device_error() & 16


def test_quantize_then_gemv_on_one_stream():
    """Requantize bf16 weights on the device, then run the GEMV on them in the
    same stream: the outputs equal the GEMV of the oracle-quantized weights."""
    N, K, n = 512, 1024, 4
    wb = synth.to_bf16_bits(synth.weights_f32(N, K, seed=9))
    x = synth.activations_bf16(n, K, seed=10)
    xt = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    wt = torch.from_numpy(wb.view(np.int16)).cuda().view(torch.bfloat16)
    packed, scale, g = nv.nvfp4_quantize_bf16(wt)
    y = nv.nvfp4_gemv_batched(packed, scale, g, xt)
    rp, rs, rg = oracle.quantize(bf16_bits_to_f32(wb))
    dev = (torch.from_numpy(rp).cuda(), torch.from_numpy(rs).cuda(),
           torch.tensor([rg], dtype=torch.float32, device="cuda"), xt)
    y_ref = nv.nvfp4_gemv_batched(*dev)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))
    assert nv.nvfp4_device_error() == 0


def test_bf16_entry_rejects_other_dtypes():
    with pytest.raises(ValueError):
        nv.nvfp4_quantize_bf16(torch.zeros(2, 16, device="cuda"))
