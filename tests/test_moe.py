"""GPU parity of the grouped read-once expert GEMV (nvfp4_moe_gemv_grouped)
against the oracle (per assignment, the expert's projection of its token).

Tolerance as for the GEMV: |y_gpu - y_ref| <= 1e-2 * (|y_ref| + 1).
Inputs: expert weights ~ N(0, 0.02) quantized by the oracle (one tensor per
expert), X ~ N(0, 1) bf16, seeded random top-k routing sorted by expert.
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


def experts(E, N, K, seed, swiglu=False):
    packs, scales, gs = [], [], []
    for e in range(E):
        if swiglu:
            w = np.empty((N, K), dtype=np.float32)
            w[0::2] = synth.weights_f32(N // 2, K, seed + 2 * e)
            w[1::2] = synth.weights_f32(N // 2, K, seed + 2 * e + 1)
        else:
            w = synth.weights_f32(N, K, seed + e)
        p, s, g = oracle.quantize(w)
        packs.append(p); scales.append(s); gs.append(g)
    return np.stack(packs), np.stack(scales), np.array(gs, dtype=np.float32)


def routing(n, E, topk, seed, force=None):
    """Seeded top-k routing (distinct experts per token), sorted by expert (stable)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    pairs = []
    for t in range(n):
        for e in rng.choice(E, size=topk, replace=False):
            pairs.append((int(e), t))
    if force is not None:
        pairs += force
    pairs.sort(key=lambda p: p[0])
    off = np.zeros(E + 1, dtype=np.int32)
    for e, _ in pairs:
        off[e + 1] += 1
    off = np.cumsum(off).astype(np.int32)
    tok = np.array([t for _, t in pairs], dtype=np.int32)
    return off, tok


def to_dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return t


def dev_x(x16):
    return torch.from_numpy(np.ascontiguousarray(x16).view(np.int16)).cuda().view(torch.bfloat16)


def host_bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def assert_close(got16, ref64):
    got = torch.from_numpy(got16.view(np.int16)).view(torch.bfloat16).double().numpy()
    err = np.abs(got - ref64)
    bad = ~(err <= TOL * (np.abs(ref64) + 1.0))
    assert not bad.any(), f"{bad.sum()} of {bad.size} out of tolerance; worst {err.max()}"


def run(packed, scale, g, x, off, tok, swiglu=False):
    y = nv.nvfp4_moe_gemv_grouped(to_dev(packed), to_dev(scale), to_dev(g), dev_x(x), to_dev(off), to_dev(tok),
                                  swiglu=swiglu)
    torch.cuda.synchronize()
    return host_bits(y)


@pytest.mark.parametrize("E,N,K,n,topk,swiglu", [
    # K % 256 == 0: the streaming tensor-core kernel
    (8, 256, 512, 4, 2, False), (16, 320, 1024, 16, 4, False), (8, 256, 2048, 12, 3, True),
    (4, 96, 4096, 3, 2, False), (3, 48, 5632, 18, 2, False),
    (24, 1536, 2048, 16, 8, True), (24, 2048, 768, 16, 8, False),   # the bench's expert shapes
    (5, 16, 7168, 20, 2, True),                                      # deepest K: fewer staged tokens per pass
    # other K: the SIMT kernel
    (6, 128, 800, 7, 2, False), (4, 64, 352, 5, 3, True)])
def test_grouped_matches_oracle(E, N, K, n, topk, swiglu):
    packed, scale, g = experts(E, N, K, seed=N + K, swiglu=swiglu)
    x = synth.activations_bf16(n, K, seed=5)
    off, tok = routing(n, E, topk, seed=E + n)
    y = run(packed, scale, g, x, off, tok, swiglu)
    y64, _ = oracle.moe_grouped(packed, scale, g, x, off, tok, swiglu=swiglu)
    assert_close(y, y64)
    assert nv.nvfp4_device_error() == 0


def test_expert_with_more_than_one_pass_of_tokens_and_empty_experts():
    E, N, K, n = 6, 128, 512, 24
    packed, scale, g = experts(E, N, K, seed=9)
    x = synth.activations_bf16(n, K, seed=10)
    # every token on expert 2 (24 > 16 tokens: two passes), experts 0, 4, 5 empty
    off, tok = routing(0, E, 1, seed=1, force=[(2, t) for t in range(n)] + [(3, 7), (1, 3)])
    y = run(packed, scale, g, x, off, tok)
    y64, _ = oracle.moe_grouped(packed, scale, g, x, off, tok)
    assert_close(y, y64)


def test_token_result_does_not_depend_on_its_expert_mates():
    E, N, K, n = 4, 256, 1024, 12
    packed, scale, g = experts(E, N, K, seed=13)
    x = synth.activations_bf16(n, K, seed=14)
    off, tok = routing(n, E, 2, seed=15)
    y = run(packed, scale, g, x, off, tok)
    # assignment j alone: its expert only, one token
    for j in range(0, len(tok), 5):
        e = int(np.searchsorted(off, j, side="right") - 1)
        off1 = np.zeros(E + 1, dtype=np.int32)
        off1[e + 1:] = 1
        y1 = run(packed, scale, g, x, off1, tok[j:j + 1].copy())
        assert np.array_equal(y1[0], y[j]), j


def test_bad_routing_sets_the_error_word():
    E, N, K, n = 2, 64, 256, 3
    packed, scale, g = experts(E, N, K, seed=17)
    x = synth.activations_bf16(n, K, seed=18)
    off = np.array([0, 2, 3], dtype=np.int32)
    tok = np.array([0, 7, 1], dtype=np.int32)     # token 7 does not exist
    run(packed, scale, g, x, off, tok)
    assert nv.nvfp4_device_error() & 32
    off_bad = np.array([0, 5, 3], dtype=np.int32)  # decreasing, past A
    run(packed, scale, g, x, off_bad, np.array([0, 1, 2], dtype=np.int32))
    assert nv.nvfp4_device_error() & 32
