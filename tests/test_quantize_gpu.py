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


def boundary_matrix(amax, bf16, seed):
    """Weights placed on and a few ulps around every E2M1 decision point
    T * d (T in 0.25, 0.75, ..., 5; d the block's fp32 divisor) for blocks
    with a spread of scales, so each code decision is as close as the format
    allows.  d and g are computed as the quantizer defines them (fp32 steps,
    scale codes from the oracle's E4M3 encoder)."""
    f32 = np.float32
    rng = np.random.Generator(np.random.PCG64(seed))
    N, K = 48, 16 * 32
    w = np.zeros((N, K), dtype=f32)
    g = f32(amax) / f32(2688.0)
    thresholds = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    for r in range(N):
        for b in range(K // 16):
            B = f32(amax * 2.0 ** rng.uniform(-14, 0))
            if bf16:
                B = bf16_bits_to_f32(synth.to_bf16_bits(np.array([B], dtype=f32)))[0]
            s_val = f32(oracle.e4m3_decode(oracle.e4m3_encode(float(B / (f32(6.0) * g)))))
            d = s_val * g
            vals = []
            for t in thresholds:
                x = np.float64(t) * np.float64(d)          # exact decision point
                if bf16:
                    u = int(synth.to_bf16_bits(np.array([x], dtype=f32))[0])
                    vals += [bf16_bits_to_f32(np.array([u + k], dtype=np.uint16))[0] for k in (-1, 0, 1)]
                else:
                    c = f32(x)
                    vals += [np.nextafter(c, f32(0)), c, np.nextafter(c, f32(np.inf))]
            pick = rng.choice(len(vals), size=15, replace=False)
            blk = np.array([vals[i] for i in pick], dtype=f32)
            blk = np.where(blk < B, blk, f32(0.0))       # keep B the block maximum
            signs = np.where(rng.random(15) < 0.5, f32(-1.0), f32(1.0))
            w[r, b * 16:b * 16 + 15] = blk * signs
            w[r, b * 16 + 15] = B
    w[0, 15] = f32(amax)
    return w


@pytest.mark.parametrize("amax", [1.0, 0.7371, 313.25])
def test_decision_boundaries_fp32(amax):
    w = boundary_matrix(amax, bf16=False, seed=int(amax * 100))
    assert_same(w, gpu_quantize(w))


@pytest.mark.parametrize("amax", [1.0, 0.7371])
def test_decision_boundaries_bf16(amax):
    wb = synth.to_bf16_bits(boundary_matrix(amax, bf16=True, seed=int(amax * 100) + 1))
    assert_same(bf16_bits_to_f32(wb), gpu_quantize(wb))


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
