"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Tolerance on bf16 outputs: |y_gpu - y_ref| <= 1e-2 * (|y_ref| + 1), with y_ref
the oracle's unrounded fp64 value.  Within one variant a batched call equals
the n single-token calls bit for bit (atlas #266, "Correctness argument").
Inputs: oracle-quantized W ~ N(0, 0.02), X ~ N(0, 1) bf16 (synth.py).
"""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

import nvfp4_weight_quantized_gemv_gb300 as nv
import oracle
import synth

pytestmark = pytest.mark.gpu
TOL = 1e-2
VARIANTS = {"fp4": nv.VARIANT_FP4, "tc": nv.VARIANT_TC, "mma": nv.VARIANT_MMA, "simt": nv.VARIANT_SIMT,
            "generic": nv.VARIANT_GENERIC}


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


def gpu_gemv(dev, variant=0, tiling=0, **kw):
    wp, ws, gs, xt = dev
    y = nv.nvfp4_gemv_batched_ex(wp, ws, gs, xt, variant=variant, tiling=tiling, **kw)
    torch.cuda.synchronize()
    return y.view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_to_f64(y16):
    return torch.from_numpy(np.ascontiguousarray(y16).view(np.int16)).view(torch.bfloat16).double().numpy()


def assert_close(y16, y64):
    yv = bf16_to_f64(y16)
    err = np.abs(yv - y64)
    bound = TOL * (np.abs(y64) + 1.0)
    bad = ~(err <= bound)
    assert not bad.any(), f"{bad.sum()} outputs out of tolerance; worst err {err.max()} at {np.argmax(err)}"


# ------------------------------------------------------------ small, full
@pytest.mark.parametrize("variant", list(VARIANTS))
@pytest.mark.parametrize("tiling", [nv.TILING_ONE_PASS, nv.TILING_GREEDY_321])
def test_tiny_workload_full_output(variant, tiling):
    # N=256, K=512, n=3 tokens, W seed 0, X seed 0
    packed, scale, g, x = make_case(256, 512, 3, 0, 0)
    y64, _ = oracle.gemv(packed, scale, g, x)
    y16 = gpu_gemv(to_gpu(packed, scale, g, x), VARIANTS[variant], tiling)
    assert_close(y16, y64)


@pytest.mark.parametrize("variant", list(VARIANTS))
@pytest.mark.parametrize("N,K,n", [(1000, 1024, 5), (200, 512, 16), (129, 256, 9), (1, 256, 1), (384, 2048, 8), (256, 8192, 16)])
def test_ragged_shapes_full_output(variant, N, K, n):
    packed, scale, g, x = make_case(N, K, n, 3, 4, outlier=0.01)
    y64, _ = oracle.gemv(packed, scale, g, x)
    y16 = gpu_gemv(to_gpu(packed, scale, g, x), VARIANTS[variant])
    assert_close(y16, y64)


def test_one_hot_pins_nibble_order_and_scale_placement():
    """Single-term outputs are exact: y[t, r] = bf16(E2M1 * E4M3 * g) at k_t.
    (FP4 variant: x = 1 expands to the single code 6 with s_0 = fl(1/6); the
    product fl(1/6) * 6 * w is w to within 2^-25 relative, below half an fp32
    ulp, so the accumulator holds w exactly as in the other kernels.)"""
    N, K = 128, 256
    packed, scale, g, _ = make_case(N, K, 1, 9, 0)
    for variant in ("fp4", "tc", "mma", "simt"):
        for k0 in range(0, K, 16):
            x = np.zeros((16, K), dtype=np.uint16)
            x[np.arange(16), k0 + np.arange(16)] = 0x3F80
            _, want = oracle.gemv(packed, scale, g, x)
            got = gpu_gemv(to_gpu(packed, scale, g, x), VARIANTS[variant])
            assert np.array_equal(got, want), (variant, k0)


# ----------------------------------------------------------- invariants
@pytest.mark.parametrize("variant", list(VARIANTS))
def test_batched_equals_single_token_calls(variant):
    N, K, n = 1536, 2048, 16
    packed, scale, g, x = make_case(N, K, n, 5, 6)
    full = gpu_gemv(to_gpu(packed, scale, g, x), VARIANTS[variant])
    for t in range(n):
        one = gpu_gemv(to_gpu(packed, scale, g, x[t:t + 1]), VARIANTS[variant])
        assert np.array_equal(one[0], full[t]), t
    greedy = gpu_gemv(to_gpu(packed, scale, g, x), VARIANTS[variant], nv.TILING_GREEDY_321)
    assert np.array_equal(greedy, full)


def test_repeat_calls_are_bit_identical():
    packed, scale, g, x = make_case(2048, 1536, 7, 1, 2)
    dev = to_gpu(packed, scale, g, x)
    first = gpu_gemv(dev)
    for _ in range(3):
        assert np.array_equal(gpu_gemv(dev), first)


@pytest.mark.parametrize("variant", [
    "fp4",
    # Known defect: on GB300 the tcgen05 f16 kernel showed rare run-to-run
    # differences in a few row blocks with long unit ranges per CTA (its
    # cause is not found); AUTO does not choose it where the FP4 kernel runs.
    pytest.param("tc", marks=pytest.mark.xfail(strict=False, reason="tcgen05 f16 kernel: rare run-to-run "
                                                                    "differences with long unit ranges")),
])
@pytest.mark.parametrize("n,num_ctas", [(16, 38), (16, 0), (4, 38)])
def test_long_unit_ranges_are_deterministic(variant, n, num_ctas):
    """Deep K and few CTAs: every CTA streams tens of units over several row
    blocks and the ring wraps many times.  Repeated calls agree bit for bit
    and with the oracle (a race between the ring stages and the hand-offs
    would show as run-to-run differences here)."""
    N, K = 14336, 10240
    packed, scale, g, x = make_case(N, K, n, 40, 41)
    dev = to_gpu(packed, scale, g, x)
    runs = [gpu_gemv(dev, VARIANTS[variant], num_ctas=num_ctas) for _ in range(6)]
    for r in runs[1:]:
        assert np.array_equal(r, runs[0])
    toks, rows = sample_points(n, N, K, 300, 42)
    ref64, _ = oracle.gemv_points(packed, scale, g, x, toks, rows)
    assert_close(runs[0][toks, rows], ref64)


@pytest.mark.parametrize("variant,num_ctas,stages", [
    (v, c, s) for v in ("fp4", "tc", "mma") for (c, s) in [(1, 2), (3, 0), (7, 4), (0, 2), (150, 8), (0, 6)]
] + [("mma", 7, 3), ("mma", 5, 5), ("fp4", 5, 3), ("fp4", 0, 10), ("fp4", 9, 11)])
def test_grid_and_ring_options(variant, num_ctas, stages):
    packed, scale, g, x = make_case(700, 1280, 4, 7, 8)
    y64, _ = oracle.gemv(packed, scale, g, x)
    y16 = gpu_gemv(to_gpu(packed, scale, g, x), VARIANTS[variant], num_ctas=num_ctas, stages=stages)
    assert_close(y16, y64)


@pytest.mark.parametrize("variant", ["fp4", "tc"])
@pytest.mark.parametrize("N,K,n,num_ctas", [
    (2000, 256, 4, 5),     # one unit per row block: every segment has one unit, two issuers idle
    (1000, 512, 9, 3),     # segments of two units
    (1000, 768, 16, 4),    # segments of three units, one per issuer
    (3000, 1280, 2, 11),   # segments of five units, split row blocks
    (640, 8192, 3, 7),     # few row blocks, every one split over several CTAs
])
def test_short_segments(variant, N, K, n, num_ctas):
    """Row-block segments shorter than the issuer rotation (tensor-memory kernels)."""
    packed, scale, g, x = make_case(N, K, n, 12, 13)
    y64, _ = oracle.gemv(packed, scale, g, x)
    assert_close(gpu_gemv(to_gpu(packed, scale, g, x), VARIANTS[variant], num_ctas=num_ctas), y64)


@pytest.mark.parametrize("num_ctas", [16, 24, 32, 48, 40])
@pytest.mark.parametrize("n", [1, 5, 16, 20])
def test_row_blocks_split_evenly(num_ctas, n):
    """8 row blocks of 12 units on 8 p CTAs (p = 2, 3, 4, 6): each row block's
    p parts are summed in a cluster of p CTAs, in CTA order; 40 CTAs split
    rows unevenly and sum through the workspace.  n = 20 takes two passes.
    Parity with the oracle, repeatability, and batched == single-token calls
    bit for bit."""
    N, K = 1024, 3072
    packed, scale, g, x = make_case(N, K, n, wseed=11, xseed=12)
    dev = to_gpu(packed, scale, g, x)
    y = gpu_gemv(dev, nv.VARIANT_FP4, num_ctas=num_ctas)
    y64, _ = oracle.gemv(packed, scale, g, x)
    assert_close(y, y64)
    assert np.array_equal(gpu_gemv(dev, nv.VARIANT_FP4, num_ctas=num_ctas), y)
    wp, ws, gs, xt = dev
    for t in range(n):
        yt = gpu_gemv((wp, ws, gs, xt[t:t + 1].contiguous()), nv.VARIANT_FP4, num_ctas=num_ctas)
        assert np.array_equal(yt[0], y[t]), t


def test_chained_calls_read_the_previous_output():
    """Back-to-back calls on one stream where call 2 reads call 1's output as X:
    the second kernel may start early (programmatic dependent launch) but must
    read X and reuse the workspace only after the first has finished."""
    p1, s1, g1, x = make_case(4096, 5120, 4, 20, 21)
    p2, s2, g2, _ = make_case(2048, 4096, 1, 22, 23)
    wp1, ws1, gs1, xt = to_gpu(p1, s1, g1, x)
    wp2, ws2, gs2, _ = to_gpu(p2, s2, g2, x[:, :4096])
    for _ in range(3):
        y1 = nv.nvfp4_gemv_batched(wp1, ws1, gs1, xt)
        y2 = nv.nvfp4_gemv_batched(wp2, ws2, gs2, y1)          # no synchronization in between
        y3 = nv.nvfp4_gemv_batched(wp1, ws1, gs1, xt)
        torch.cuda.synchronize()
        y1h = y1.view(torch.int16).cpu().numpy().view(np.uint16)
        y64, _ = oracle.gemv(p1, s1, g1, x)
        assert_close(y1h, y64)
        assert np.array_equal(y3.view(torch.int16).cpu().numpy(), y1.view(torch.int16).cpu().numpy())
        y2_sync = nv.nvfp4_gemv_batched(wp2, ws2, gs2, y1)
        torch.cuda.synchronize()
        assert np.array_equal(y2.view(torch.int16).cpu().numpy(), y2_sync.view(torch.int16).cpu().numpy())


def test_chained_calls_with_every_row_block_whole():
    """As above, with a first call whose partition gives every CTA exactly one
    whole row block (N = 152 row blocks, K = one unit): nothing is left for
    the reduction kernel, which must still not complete before the GEMV."""
    N1, K1 = 152 * 128, 256
    plan = nv.nvfp4_gemv_plan(2, N1, K1)
    if plan["variant"] not in ("fp4", "tc") or plan["num_ctas"] != 152:
        pytest.skip("needs a tensor-memory path on a 152-SM part")
    p1, s1, g1, x = make_case(N1, K1, 2, 30, 31)
    p2, s2, g2, _ = make_case(256, N1, 2, 32, 33)
    wp1, ws1, gs1, xt = to_gpu(p1, s1, g1, x)
    wp2, ws2, gs2, _ = to_gpu(p2, s2, g2, synth.activations_bf16(2, N1, 34))
    y1_ref, _ = oracle.gemv(p1, s1, g1, x)
    for _ in range(5):
        y1 = nv.nvfp4_gemv_batched(wp1, ws1, gs1, xt)
        y2 = nv.nvfp4_gemv_batched(wp2, ws2, gs2, y1)          # no synchronization in between
        torch.cuda.synchronize()
        y1h = y1.view(torch.int16).cpu().numpy().view(np.uint16)
        assert_close(y1h, y1_ref)
        y2_ref, _ = oracle.gemv(p2, s2, g2, y1h)
        assert_close(y2.view(torch.int16).cpu().numpy().view(np.uint16), y2_ref)


def test_generic_paths_for_unaligned_or_ragged_k():
    # K % 256 != 0 -> generic kernel
    packed, scale, g, x = make_case(300, 784, 3, 2, 3)
    y64, _ = oracle.gemv(packed, scale, g, x)
    assert_close(gpu_gemv(to_gpu(packed, scale, g, x)), y64)
    # misaligned activation pointer -> generic kernel, same answer
    packed, scale, g, x = make_case(256, 512, 2, 2, 3)
    wp, ws, gs, _ = to_gpu(packed, scale, g, x)
    buf = torch.zeros(2 * 512 + 8, dtype=torch.int16, device="cuda")
    buf[1:1 + 2 * 512] = torch.from_numpy(x.view(np.int16).ravel()).cuda()
    xt = buf[1:1 + 2 * 512].view(torch.bfloat16).view(2, 512)
    y = nv.nvfp4_gemv_batched(wp, ws, gs, xt)
    torch.cuda.synchronize()
    y64, _ = oracle.gemv(packed, scale, g, x)
    assert_close(y.view(torch.int16).cpu().numpy().view(np.uint16), y64)


def test_more_than_16_tokens_and_noop():
    packed, scale, g, x = make_case(512, 1024, 21, 4, 5)
    y64, _ = oracle.gemv(packed, scale, g, x)
    dev = to_gpu(packed, scale, g, x)
    assert_close(gpu_gemv(dev), y64)
    wp, ws, gs, xt = dev
    y = torch.full((0, 512), 7.0, dtype=torch.bfloat16, device="cuda")
    nv.nvfp4_gemv_batched(wp, ws, gs, xt[:0].contiguous(), y)


def test_output_guard_bands_untouched():
    N, K, n = 333, 512, 5
    packed, scale, g, x = make_case(N, K, n, 6, 7)
    wp, ws, gs, xt = to_gpu(packed, scale, g, x)
    pad = 64
    buf = torch.full((n * N + 2 * pad,), 12345, dtype=torch.int16, device="cuda")
    y = buf[pad:pad + n * N].view(torch.bfloat16).view(n, N)
    for variant in VARIANTS.values():
        nv.nvfp4_gemv_batched_ex(wp, ws, gs, xt, y, variant=variant)
        torch.cuda.synchronize()
        b = buf.cpu().numpy()
        assert np.all(b[:pad] == 12345) and np.all(b[pad + n * N:] == 12345)


def test_caller_workspace():
    packed, scale, g, x = make_case(1024, 2048, 3, 8, 9)
    wp, ws, gs, xt = to_gpu(packed, scale, g, x)
    nbytes = nv.nvfp4_gemv_workspace_size(3, 1024, 2048)
    work = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    y = nv.nvfp4_gemv_batched_ex(wp, ws, gs, xt, workspace=work)
    y2 = nv.nvfp4_gemv_batched_ex(wp, ws, gs, xt, workspace=work)
    torch.cuda.synchronize()
    assert torch.equal(y, y2)
    y64, _ = oracle.gemv(packed, scale, g, x)
    assert_close(y.view(torch.int16).cpu().numpy().view(np.uint16), y64)
    small = torch.zeros(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(nv.Nvfp4Error):
        nv.nvfp4_gemv_batched_ex(wp, ws, gs, xt, workspace=small)


def test_activation_beyond_f16_range_is_rescaled():
    packed, scale, g, x = make_case(256, 1024, 4, 1, 1)
    xf = synth.activations_f32(4, 1024, 1)
    xf[1, 17] = 3.0e5            # beyond f16's range
    xf[2, 900] = -1.0e6
    x = synth.to_bf16_bits(xf)
    y64, _ = oracle.gemv(packed, scale, g, x)
    for variant in VARIANTS:
        assert_close(gpu_gemv(to_gpu(packed, scale, g, x), VARIANTS[variant]), y64)


# Variants that take bf16 activations over their whole range (the FP4 kernel's
# per-row term scales, the generic kernel's fp32 FMAs); the others convert X to
# f16 and are in range only for 2^-6 <= |x| < 1.68e7 or so.
FULL_RANGE_X = ("fp4", "generic")


@pytest.mark.parametrize("x_max", [1.6e7, 2.0 ** -18, 1.0e-30])
def test_activation_magnitudes(x_max):
    """Rows scaled to max|x| = x_max (up to 1.6e7, just inside the f16 x 2^-8
    range of the tcgen05 kernel; down to 1e-30), next to an all-zero row and a
    row with one non-zero entry.  Tolerance relative to each row's own output
    scale: |y - y_ref| <= 1e-2 * (|y_ref| + max_r |y_ref|) per token."""
    N, K, n = 384, 1536, 4
    packed, scale, g, _ = make_case(N, K, n, 14, 15)
    xf = synth.activations_f32(n, K, 16).astype(np.float64)
    xf *= x_max / np.abs(xf).max()
    xf[1] = 0.0
    xf[2] = 0.0
    xf[2, 700] = -x_max
    x = synth.to_bf16_bits(xf.astype(np.float32))
    y64, _ = oracle.gemv(packed, scale, g, x)
    row_scale = np.abs(y64).max(axis=1, keepdims=True)
    for variant in (VARIANTS if x_max >= 1.0 else FULL_RANGE_X):
        yv = bf16_to_f64(gpu_gemv(to_gpu(packed, scale, g, x), VARIANTS[variant]))
        assert np.all(yv[1] == 0.0), variant
        err = np.abs(yv - y64)
        assert np.all(err <= TOL * (np.abs(y64) + row_scale)), (variant, (err / row_scale).max())
    assert nv.nvfp4_device_error() == 0


def test_nan_scale_propagates():
    packed, scale, g, x = make_case(256, 512, 2, 1, 1)
    scale = scale.copy()
    scale[10, 3] = 0x7F
    y64, _ = oracle.gemv(packed, scale, g, x)
    for variant in VARIANTS.values():
        y16 = gpu_gemv(to_gpu(packed, scale, g, x), variant)
        yv = bf16_to_f64(y16)
        assert np.all(np.isnan(yv[:, 10])) and np.all(np.isnan(y64[:, 10]))
        keep = np.ones(256, bool)
        keep[10] = False
        assert_close(y16[:, keep], y64[:, keep])


# --------------------------------------------------- full-size workloads
def sample_points(n, N, K, count, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    rows = np.concatenate([[0, 1, 127, 128, N - 129, N - 128, N - 1], rng.integers(0, N, count)])
    toks = rng.integers(0, n, rows.shape[0])
    return toks, rows


@pytest.mark.parametrize("name,N,K,ns,outlier", [
    ("attn_qkv", 14336, 5120, (1, 2, 3, 4), 0.0),
    ("o_proj", 5120, 6144, (8,), 0.01),
    ("fused_qkv", 16384, 5120, (16,), 0.0),
])
def test_full_size_workloads_sampled(name, N, K, ns, outlier):
    w = synth.weights_f32(N, K, 0)
    packed, scale, g = oracle.quantize(w)
    nmax = max(ns)
    x = synth.activations_bf16(nmax, K, 1, outlier)
    wp, ws, gs, xt_all = to_gpu(packed, scale, g, x)
    per_token = {}
    for n in ns:
        y = nv.nvfp4_gemv_batched(wp, ws, gs, xt_all[:n].contiguous())
        torch.cuda.synchronize()
        y16 = y.view(torch.int16).cpu().numpy().view(np.uint16)
        assert not np.isnan(bf16_to_f64(y16)).any()
        toks, rows = sample_points(n, N, K, 400, 11 + n)
        ref64, _ = oracle.gemv_points(packed, scale, g, x[:n], toks, rows)
        assert_close(y16[toks, rows], ref64)
        per_token[n] = y16
    # batched == single token, bit for bit, on the full-size launch configuration
    if 1 in per_token:
        for n, y16 in per_token.items():
            assert np.array_equal(y16[0], per_token[1][0])
    else:
        y1 = nv.nvfp4_gemv_batched(wp, ws, gs, xt_all[nmax - 1:nmax].contiguous())
        torch.cuda.synchronize()
        assert np.array_equal(y1.view(torch.int16).cpu().numpy().view(np.uint16)[0], per_token[nmax][nmax - 1])


def oracle_rows_parallel(packed, scale, g, x):
    """The oracle's full output, its rows split over the host cores (the oracle's
    C routine runs without the interpreter lock, so threads run in parallel)."""
    from concurrent.futures import ThreadPoolExecutor
    N = packed.shape[0]
    cores = os.cpu_count() or 1
    bounds = np.linspace(0, N, min(cores, N) + 1).astype(int)

    def part(i):
        r0, r1 = bounds[i], bounds[i + 1]
        return oracle.gemv(np.ascontiguousarray(packed[r0:r1]), np.ascontiguousarray(scale[r0:r1]), g, x)[0]
    with ThreadPoolExecutor(len(bounds) - 1) as ex:
        return np.concatenate(list(ex.map(part, range(len(bounds) - 1))), axis=1)


@pytest.mark.parametrize("name,N,K,n", [("attn_qkv", 14336, 5120, 4), ("fused_qkv", 16384, 5120, 16)])
def test_full_size_whole_output(name, N, K, n):
    """Every output of a full-size call against the oracle, in the launch
    configuration the benchmark times (AUTO plan, one CTA per SM)."""
    packed, scale, g = oracle.quantize(synth.weights_f32(N, K, 0))
    x = synth.activations_bf16(n, K, 1)
    y16 = gpu_gemv(to_gpu(packed, scale, g, x))
    assert_close(y16, oracle_rows_parallel(packed, scale, g, x))


def test_decode_step_chain_of_32_calls():
    """Sixteen layers of qkv (N=14336, K=5120) then o_proj (N=5120, K=6144) on one
    stream with no synchronization: o_proj reads the first 6144 qkv outputs,
    the next layer's qkv reads the o_proj output.  Each call is then checked on
    sampled points against the oracle given the GPU's own input to that call."""
    n = 8
    layers = 16
    mats = {}
    for name, (N, K) in (("qkv", (14336, 5120)), ("o", (5120, 6144))):
        mats[name] = []
        for i in range(4):
            packed, scale, g = oracle.quantize(synth.weights_f32(N, K, 50 + 10 * i + (name == "o")))
            mats[name].append((packed, scale, g, to_gpu(packed, scale, g, np.zeros((1, K), np.uint16))[:3]))
    x0 = synth.activations_bf16(n, 5120, 60)
    x = torch.from_numpy(x0.view(np.int16)).cuda().view(torch.bfloat16)
    outs = []
    for layer in range(layers):
        wq = mats["qkv"][layer % 4]
        yq = nv.nvfp4_gemv_batched(*wq[3], x)
        xo = yq[:, :6144].contiguous()
        wo = mats["o"][layer % 4]
        yo = nv.nvfp4_gemv_batched(*wo[3], xo)
        outs.append((wq, x, yq))
        outs.append((wo, xo, yo))
        x = yo
    torch.cuda.synchronize()
    for i, ((packed, scale, g, _), xin, y) in enumerate(outs):
        xin16 = xin.view(torch.int16).cpu().numpy().view(np.uint16)
        y16 = y.view(torch.int16).cpu().numpy().view(np.uint16)
        nn, N = y16.shape
        toks, rows = sample_points(nn, N, packed.shape[1] * 2, 100, 70 + i)
        ref64, _ = oracle.gemv_points(packed, scale, g, xin16, toks, rows)
        assert_close(y16[toks, rows], ref64)
    assert nv.nvfp4_device_error() == 0


def test_no_device_error_recorded():
    assert nv.nvfp4_device_error() == 0
