"""Pins for the CPU oracle (oracle/), independent of the oracle's own code.

Each test checks the oracle against something other than itself: the code
tables of the OCP FP4 E2M1 / E4M3 definitions, torch's float8_e4m3fn and
bfloat16 conversions (library routines), searches over every representable
value, hand-worked golden cases (tests/golden/), a dense numpy float64
reconstruction, and invariants of the projection.  None of them needs a GPU.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth
from golden_io import fractions, hex_bytes, read_cases

# FP4 E2M1 code table (OCP Microscaling Formats v1.0): codes 0..7 are the
# non-negative magnitudes, codes 8..15 the same magnitudes negated.
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def e4m3_library_values():
    """All 256 E4M3 codes decoded by torch's float8_e4m3fn."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def bf16_library_values():
    """All 65536 bf16 bit patterns decoded by torch."""
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    return bits.view(torch.bfloat16).to(torch.float64).numpy()


# --------------------------------------------------------------------- codecs
def test_e2m1_decode_matches_code_table():
    for code in range(16):
        mag = E2M1_TABLE[code & 7]
        v = oracle.e2m1_decode(code)
        assert v == (-mag if code & 8 else mag)
        assert math.copysign(1.0, v) == (-1.0 if code & 8 else 1.0)


def test_e4m3_decode_matches_torch_for_all_codes():
    ref = e4m3_library_values()
    for code in range(256):
        v = oracle.e4m3_decode(code)
        if math.isnan(ref[code]):
            assert math.isnan(v), code
        else:
            assert v == ref[code], (code, v, ref[code])
    # the largest finite code is 448 and 0x7F / 0xFF are NaN
    assert oracle.e4m3_decode(0x7E) == 448.0
    assert math.isnan(oracle.e4m3_decode(0x7F)) and math.isnan(oracle.e4m3_decode(0xFF))


def _nearest_even_code(value, table_codes, table_vals):
    """Argmin over a code table; ties go to the even code (even mantissa)."""
    best = None
    for c, tv in zip(table_codes, table_vals):
        d = abs(Fraction(value) - Fraction(tv))
        if best is None or d < best[0] or (d == best[0] and c % 2 == 0 and best[1] % 2 == 1):
            best = (d, c)
    return best[1]


def test_e4m3_encode_is_nearest_even_with_saturation():
    lib = e4m3_library_values()
    codes = [c for c in range(0x7F)]            # 0x00..0x7E: non-negative finite codes
    vals = [lib[c] for c in codes]
    rng = np.random.Generator(np.random.PCG64(7))
    samples = list(rng.uniform(0, 460, 400).astype(np.float32))
    samples += list((2.0 ** rng.uniform(-12, 9, 400)).astype(np.float32))
    # exact midpoints between neighbouring codes (ties) and the codes themselves
    for a, b in zip(vals[:-1], vals[1:]):
        samples += [np.float32(a), np.float32((a + b) / 2)]
    for s in samples:
        s = float(s)
        want = 0x7E if s >= 448.0 else _nearest_even_code(s, codes, vals)
        assert oracle.e4m3_encode(s) == want, s


def test_e4m3_encode_agrees_with_torch_cast_in_range():
    rng = np.random.Generator(np.random.PCG64(8))
    v = (2.0 ** rng.uniform(-11, 8.8, 2000)).astype(np.float32)
    v = v[v <= 448.0]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(x)) for x in v], dtype=np.uint8)
    assert np.array_equal(got, ref)


def test_e2m1_encode_is_nearest_even_with_saturation():
    codes = list(range(8))
    rng = np.random.Generator(np.random.PCG64(9))
    samples = list(rng.uniform(-7, 7, 2000))
    ties = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    samples += ties + [-t for t in ties] + E2M1_TABLE + [-v for v in E2M1_TABLE] + [6.5, -100.0]
    for v in samples:
        mag = 7 if abs(v) >= 6.0 else _nearest_even_code(abs(v), codes, E2M1_TABLE)
        want = 0 if mag == 0 else (mag | 8 if v < 0 else mag)
        assert oracle.e2m1_encode(v) == want, v
    # the tie table, stated by value
    expect = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0}
    for v, r in expect.items():
        assert oracle.e2m1_decode(oracle.e2m1_encode(v)) == r


def _bf16_by_search(v, lib_sorted, lib_bits_sorted):
    """Nearest bf16 to v by searching all finite positive patterns; ties to even."""
    if v == 0.0:
        return 0x8000 if math.copysign(1.0, v) < 0 else 0
    a = abs(v)
    sign = 0x8000 if v < 0 else 0
    i = int(np.searchsorted(lib_sorted, a))
    top = float(lib_sorted[-1])
    if i >= len(lib_sorted):
        # above the largest finite value: rounds to it unless past the half-ulp
        half_ulp = Fraction(2) ** 127 * Fraction(1, 2 ** 8)
        return sign | (0x7F80 if Fraction(a) >= Fraction(top) + half_ulp else int(lib_bits_sorted[-1]))
    hi_v, hi_b = float(lib_sorted[i]), int(lib_bits_sorted[i])
    if hi_v == a:
        return sign | hi_b
    lo_v, lo_b = float(lib_sorted[i - 1]), int(lib_bits_sorted[i - 1])
    dl, dh = Fraction(a) - Fraction(lo_v), Fraction(hi_v) - Fraction(a)
    if dl < dh or (dl == dh and lo_b % 2 == 0):
        return sign | lo_b
    return sign | hi_b


def test_bf16_encode_matches_search_over_all_patterns():
    lib = bf16_library_values()
    pos = np.arange(0x0000, 0x7F80)              # zero and positive finite patterns, increasing
    lib_sorted, bits_sorted = lib[pos], pos
    assert np.all(np.diff(lib_sorted) > 0)
    rng = np.random.Generator(np.random.PCG64(10))
    vals = list(rng.standard_normal(1500) * 10.0 ** rng.uniform(-30, 30, 1500))
    # double-rounding traps: just above/below bf16 ties, at spacings fp32 would erase
    for base in (257.0, 259.0, 1.00390625, 3.0e-39):
        for eps in (2.0 ** -20, -(2.0 ** -20), 2.0 ** -40):
            vals.append(base * (1.0 + eps))
    vals += [0.0, -0.0, 1e-45, -3e38, 3.4e38, 1e39, float(lib_sorted[0]) / 2]
    for v in vals:
        assert oracle.bf16_encode(v) == _bf16_by_search(v, lib_sorted, bits_sorted), v
    assert oracle.bf16_encode(float("inf")) == 0x7F80
    assert oracle.bf16_encode(float("-inf")) == 0xFF80
    assert oracle.bf16_encode(float("nan")) == 0x7FC0


def test_bf16_codec_agrees_with_torch_on_fp32_values():
    rng = np.random.Generator(np.random.PCG64(11))
    v = (rng.standard_normal(3000) * 10.0 ** rng.uniform(-20, 20, 3000)).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_encode(float(x)) for x in v], dtype=np.uint16)
    assert np.array_equal(got, ref)
    lib = bf16_library_values()
    for b in rng.integers(0, 65536, 500):
        d = oracle.bf16_decode(int(b))
        assert (math.isnan(d) and math.isnan(lib[b])) or d == lib[b]


# ----------------------------------------------------------------- GEMV: pins
@pytest.mark.parametrize("case", read_cases("gemv_hand_cases.txt"), ids=lambda c: c["name"])
def test_gemv_hand_worked_cases(case):
    K = int(case["K"][0])
    x = np.array([hex_bytes(case["x"])], dtype=np.uint16)
    packed = np.array([hex_bytes(case["packed"])], dtype=np.uint8)
    scale = np.array([hex_bytes(case["scale"])], dtype=np.uint8)
    assert x.shape == (1, K) and packed.shape == (1, K // 2) and scale.shape == (1, K // 16)
    g = float(case["g"][0])
    y64, y16 = oracle.gemv(packed, scale, g, x)
    want64 = float(case["y64"][0])
    if math.isnan(want64):
        assert math.isnan(y64[0, 0])
    else:
        assert y64[0, 0] == want64
    assert int(y16[0, 0]) == int(case["y16"][0], 16)


def dequant_dense(packed, scale):
    """Independent dense W[N, K] in float64: code table x torch's E4M3 decode."""
    N, half = packed.shape
    K = half * 2
    nib = np.empty((N, K), dtype=np.int64)
    nib[:, 0::2] = packed & 0x0F
    nib[:, 1::2] = packed >> 4
    mag = np.array(E2M1_TABLE)[nib & 7]
    q = np.where(nib & 8, -mag, mag)
    s = e4m3_library_values()[scale.astype(np.int64)]
    return q * np.repeat(s, 16, axis=1)


def random_nvfp4(rng, N, K):
    packed = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    scale = rng.integers(0, 0x7F, (N, K // 16), dtype=np.uint8)   # finite, non-negative
    return packed, scale


@pytest.mark.parametrize("N,K,n", [(16, 16, 1), (16, 16, 5), (8, 64, 3), (3, 128, 16)])
def test_gemv_brute_force_against_dense_reconstruction(N, K, n):
    rng = np.random.Generator(np.random.PCG64(100 + N + K + n))
    packed, scale = random_nvfp4(rng, N, K)
    x = synth.activations_bf16(n, K, seed=5)
    g = float(np.float32(rng.uniform(1e-4, 1e-2)))
    y64, y16 = oracle.gemv(packed, scale, g, x)
    xf = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    ref = (xf @ dequant_dense(packed, scale).T) * g
    np.testing.assert_allclose(y64, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    lib = bf16_library_values()
    pos = np.arange(0x0000, 0x7F80)
    for t in range(n):
        for r in range(N):
            assert int(y16[t, r]) == _bf16_by_search(float(y64[t, r]), lib[pos], pos)


def test_gemv_one_hot_recovers_each_column():
    N, K = 16, 16
    rng = np.random.Generator(np.random.PCG64(3))
    packed, scale = random_nvfp4(rng, N, K)
    W = dequant_dense(packed, scale)
    x = np.zeros((K, K), dtype=np.uint16)
    x[np.arange(K), np.arange(K)] = 0x3F80          # bf16 1.0 at position k for token k
    y64, _ = oracle.gemv(packed, scale, 1.0, x)
    assert np.array_equal(y64, W.T)                 # token k sees column k of W


def test_gemv_invariants():
    N, K, n = 24, 96, 6
    rng = np.random.Generator(np.random.PCG64(4))
    packed, scale = random_nvfp4(rng, N, K)
    x = synth.activations_bf16(n, K, seed=6)
    g = 0.0078125
    y64, y16 = oracle.gemv(packed, scale, g, x)
    # batched == n separate single-token calls, bit for bit
    for t in range(n):
        a64, a16 = oracle.gemv(packed, scale, g, x[t:t + 1])
        assert np.array_equal(a64[0], y64[t]) and np.array_equal(a16[0], y16[t])
    # permuting tokens permutes the rows of Y
    perm = rng.permutation(n)
    p64, _ = oracle.gemv(packed, scale, g, x[perm])
    assert np.array_equal(p64, y64[perm])
    # doubling g (a power of two) doubles Y exactly
    d64, d16 = oracle.gemv(packed, scale, 2 * g, x)
    assert np.array_equal(d64, 2 * y64)
    # an all-zero scale row gives a zero output row
    s0 = scale.copy()
    s0[5] = 0
    z64, z16 = oracle.gemv(packed, s0, g, x)
    assert np.all(z64[:, 5] == 0) and np.all((z16[:, 5] & 0x7FFF) == 0)
    # row and point evaluation agree with the full product
    r64, _ = oracle.gemv_rows(packed, scale, g, x, 7, 11)
    assert np.array_equal(r64[:, 7:11], y64[:, 7:11]) and np.all(r64[:, :7] == 0)
    tok, row = rng.integers(0, n, 20), rng.integers(0, N, 20)
    q64, q16 = oracle.gemv_points(packed, scale, g, x, tok, row)
    assert np.array_equal(q64, y64[tok, row]) and np.array_equal(q16, y16[tok, row])


def test_gemv_is_linear_in_x():
    # x1, x2 and x1 + x2 are small integers: all exact in bf16 and the sums are exact
    N, K = 12, 64
    rng = np.random.Generator(np.random.PCG64(12))
    packed, scale = random_nvfp4(rng, N, K)
    a = rng.integers(-8, 8, (2, K)).astype(np.float32)
    b = rng.integers(-8, 8, (2, K)).astype(np.float32)
    ya, _ = oracle.gemv(packed, scale, 1.0, synth.to_bf16_bits(a))
    yb, _ = oracle.gemv(packed, scale, 1.0, synth.to_bf16_bits(b))
    yab, _ = oracle.gemv(packed, scale, 1.0, synth.to_bf16_bits(a + b))
    assert np.array_equal(yab, ya + yb)


# ------------------------------------------------------------ quantizer: pins
@pytest.mark.parametrize("case", read_cases("quantize_hand_cases.txt"), ids=lambda c: c["name"])
def test_quantize_hand_derived_cases(case):
    N, K = int(case["N"][0]), int(case["K"][0])
    w = np.array([float(f) for f in fractions(case["w"])], dtype=np.float32).reshape(N, K)
    assert all(Fraction(float(v)) == f for v, f in zip(w.ravel(), fractions(case["w"])))
    packed, scale, g = oracle.quantize(w)
    assert Fraction(g) == Fraction(case["g"][0])
    assert scale.ravel().tolist() == hex_bytes(case["scale"])
    assert packed.ravel().tolist() == hex_bytes(case["packed"])


def test_quantize_decisions_match_argmin_restatement():
    """Every scale and element code is the nearest-even table entry, decided in fp32."""
    N, K = 16, 256
    w = synth.weights_f32(N, K, seed=21)
    w[3, 40:56] *= 1e-4                          # a block whose scale is subnormal
    w[7, 0:16] = 0.0                             # an all-zero block
    packed, scale, g = oracle.quantize(w)
    f32 = np.float32
    assert g == f32(np.abs(w).max()) / f32(2688.0)
    lib = e4m3_library_values()
    scodes = list(range(0x7F))
    svals = [lib[c] for c in scodes]
    nib = np.empty((N, K), dtype=np.int64)
    nib[:, 0::2] = packed & 0x0F
    nib[:, 1::2] = packed >> 4
    for r in range(N):
        for b in range(K // 16):
            blk = w[r, b * 16:(b + 1) * 16]
            s_f = f32(np.abs(blk).max()) / (f32(6.0) * f32(g))
            want_s = 0x7E if s_f >= 448 else _nearest_even_code(float(s_f), scodes, svals)
            assert scale[r, b] == want_s
            s_val = f32(lib[want_s])
            for j in range(16):
                code = int(nib[r, b * 16 + j])
                if s_val == 0:
                    assert code == 0
                    continue
                v = float(f32(blk[j]) / (s_val * f32(g)))
                mag = 7 if abs(v) >= 6 else _nearest_even_code(abs(v), list(range(8)), E2M1_TABLE)
                assert code == (0 if mag == 0 else (mag | 8 if v < 0 else mag)), (r, b, j)


def test_quantize_round_trip_bounds():
    N, K = 64, 512
    w = synth.weights_f32(N, K, seed=0)
    packed, scale, g = oracle.quantize(w)
    assert scale.max() <= 0x7E                   # never NaN, never above 448
    W = dequant_dense(packed, scale) * g
    s = e4m3_library_values()[scale.astype(np.int64)] * g
    s_full = np.repeat(s, 16, axis=1)
    # local E2M1 grid step: 0.5 below 2, 1 below 4, 2 above; error <= half a step
    a = np.abs(w / s_full)
    step = np.where(a < 2, 0.5, np.where(a < 4, 1.0, 2.0))
    assert np.all(np.abs(w - W) <= 0.5 * step * s_full * (1 + 1e-6) + 1e-30)
    # every decoded block max is within 6 * s * g
    blk = np.abs(W).reshape(N, K // 16, 16).max(axis=2)
    assert np.all(blk <= 6 * s * (1 + 1e-12))


def test_quantize_rejects_bad_input():
    with pytest.raises(ValueError):
        oracle.quantize(np.ones((2, 24), dtype=np.float32))
    bad = np.ones((2, 16), dtype=np.float32)
    bad[1, 3] = np.inf
    with pytest.raises(ValueError):
        oracle.quantize(bad)


# ------------------------------------------------------------------ SwiGLU
# Logistic sigmoid at a few points, from standard tables (sigma(a) = 1/(1+e^-a)).
SIGMOID_TABLE = {1.0: 0.7310585786300049, -2.0: 0.11920292202211755, 3.0: 0.9525741268224334,
                 -0.5: 0.3775406687981454, 0.0: 0.5}


def test_swiglu_matches_tabulated_sigmoid():
    gates = list(SIGMOID_TABLE)
    ups = [2.0, -1.5, 0.25, 4.0, 7.0]
    gu = np.array([[v for pair in zip(gates, ups) for v in pair]], dtype=np.float64)
    h64, h16 = oracle.swiglu(gu)
    for f, (a, u) in enumerate(zip(gates, ups)):
        assert math.isclose(h64[0, f], a * SIGMOID_TABLE[a] * u, rel_tol=1e-15, abs_tol=1e-300)
        assert h16[0, f] == oracle.bf16_encode(h64[0, f])


def test_swiglu_special_cases():
    gu = np.array([[0.0, 123.0, 5.0, 0.0, 40.0, 2.0, -40.0, 3.0, -745.0, 1.0]], dtype=np.float64)
    h64, h16 = oracle.swiglu(gu)
    assert h64[0, 0] == 0.0 and h64[0, 1] == 0.0          # gate 0 or up 0
    assert math.isclose(h64[0, 2], 80.0, rel_tol=1e-15)    # sigma(40) = 1 - 4e-18
    assert abs(h64[0, 3]) < 1e-15                          # sigma(-40) ~ 4.2e-18
    assert h64[0, 4] == 0.0 or abs(h64[0, 4]) < 1e-300     # exp overflow side: -745 / inf
    assert h16[0, 0] == 0 and h16[0, 4] in (0, 0x8000)
    assert h16[0, 3] == oracle.bf16_encode(h64[0, 3])      # tiny, still a normal bf16


def test_gemv_swiglu_interleaving_matches_two_projections():
    """Rows 2f / 2f+1 of the joint matrix are gate f / up f: the joint call
    equals the activation applied to two separate projections."""
    rng = np.random.Generator(np.random.PCG64(11))
    F, K, n = 24, 64, 3
    wg = rng.standard_normal((F, K), dtype=np.float32)
    wu = rng.standard_normal((F, K), dtype=np.float32) * np.float32(0.5)
    w = np.empty((2 * F, K), dtype=np.float32)
    w[0::2], w[1::2] = wg, wu
    packed, scale, g = oracle.quantize(w)
    x = synth.activations_bf16(n, K, seed=12)
    h64, h16 = oracle.gemv_swiglu(packed, scale, g, x)
    g64, _ = oracle.gemv(packed[0::2], scale[0::2], g, x)
    u64, _ = oracle.gemv(packed[1::2], scale[1::2], g, x)
    expect = g64 / (1.0 + np.exp(-g64)) * u64
    assert np.allclose(h64, expect, rtol=1e-13, atol=1e-13)
    # swapping the roles changes the result (silu is not symmetric)
    swapped = u64 / (1.0 + np.exp(-u64)) * g64
    assert not np.allclose(h64, swapped, rtol=1e-3, atol=1e-3)


# ----------------------------------------------------------- routed experts
def test_moe_grouped_routing_semantics():
    rng = np.random.Generator(np.random.PCG64(31))
    E, N, K, n = 3, 40, 64, 5
    ws = [oracle.quantize(rng.standard_normal((N, K), dtype=np.float32)) for _ in range(E)]
    packed = np.stack([w[0] for w in ws]); scale = np.stack([w[1] for w in ws])
    g = np.array([w[2] for w in ws], dtype=np.float32)
    x = synth.activations_bf16(n, K, seed=32)
    # expert 0: tokens 4, 1; expert 1: none; expert 2: tokens 0, 4, 2
    off = np.array([0, 2, 2, 5], dtype=np.int32)
    tok = np.array([4, 1, 0, 4, 2], dtype=np.int32)
    y64, y16 = oracle.moe_grouped(packed, scale, g, x, off, tok)
    for j, (e, t) in enumerate([(0, 4), (0, 1), (2, 0), (2, 4), (2, 2)]):
        r64, r16 = oracle.gemv(packed[e], scale[e], float(g[e]), x[t:t + 1])
        assert np.array_equal(y64[j], r64[0]) and np.array_equal(y16[j], r16[0])
    # one expert holding every token is the plain batched projection
    a64, _ = oracle.moe_grouped(packed[:1], scale[:1], g[:1], x, np.array([0, n], np.int32), np.arange(n, dtype=np.int32))
    b64, _ = oracle.gemv(packed[0], scale[0], float(g[0]), x)
    assert np.array_equal(a64, b64)
