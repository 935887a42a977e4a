"""GB300 (sm_103a) NVFP4 batched decode GEMV -- Python binding of the C ABI.

Thin ctypes marshalling over ``libnvfp4_gemv.so`` (declared in
``include/nvfp4_gemv.h``).  Functions carry the C entry points' names and
take torch tensors (device memory, streams) or numpy arrays (host quantizer);
every step of the computation runs in the library's CUDA kernels.  If the
library is missing the import of any entry point raises -- there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libnvfp4_gemv.so")
# the same library built with device index checks (buildlib.build(debug_bounds=True));
# assign it to LIB_PATH before the first call to use it
DEBUG_LIB_PATH = os.path.join(PKG, "libnvfp4_gemv_debug.so")

# nvfp4_status
NVFP4_OK = 0
NVFP4_ERR_INVALID_ARG = 1
NVFP4_ERR_MISALIGNED = 2
NVFP4_ERR_UNSUPPORTED = 3
NVFP4_ERR_CUDA = 4
NVFP4_ERR_DEVICE_TIMEOUT = 5
NVFP4_ERR_WORKSPACE = 6
NVFP4_ERR_DEVICE_INPUT = 7
NVFP4_ERR_DEVICE_BOUNDS = 8

# nvfp4_variant / nvfp4_tiling
VARIANT_AUTO, VARIANT_MMA, VARIANT_SIMT, VARIANT_GENERIC, VARIANT_TC, VARIANT_FP4 = 0, 1, 2, 3, 4, 5
TILING_AUTO, TILING_ONE_PASS, TILING_GREEDY_321 = 0, 1, 2
VARIANT_NAMES = {0: "auto", 1: "mma", 2: "simt", 3: "generic", 4: "tc", 5: "fp4"}
TILING_NAMES = {0: "auto", 1: "one_pass", 2: "greedy_321"}

# Names the C ABI exports (include/nvfp4_gemv.h).
EXPORTS = ("nvfp4_gemv_batched", "nvfp4_gemv_batched_ex", "nvfp4_gemv_batched_noalloc",
           "nvfp4_gemv_swiglu", "nvfp4_ffn_swiglu", "nvfp4_moe_gemv_grouped",
           "nvfp4_gemv_workspace_size", "nvfp4_gemv_plan",
           "nvfp4_quantize_ref", "nvfp4_quantize", "nvfp4_quantize_bf16", "nvfp4_device_error",
           "nvfp4_selftest_wait_timeout", "nvfp4_last_error", "nvfp4_version")


class Nvfp4Error(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"nvfp4 status {status}: {message}")
        self.status = status


class nvfp4_gemv_opts(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int), ("tiling", ctypes.c_int), ("num_ctas", ctypes.c_int),
                ("stages", ctypes.c_int), ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("inflight", ctypes.c_int)]


class nvfp4_gemv_plan_info(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int), ("tiling", ctypes.c_int), ("passes", ctypes.c_int),
                ("tile_tokens", ctypes.c_int * 16), ("num_ctas", ctypes.c_int), ("stages", ctypes.c_int),
                ("smem_bytes", ctypes.c_int), ("units", ctypes.c_longlong)]


_lock = threading.Lock()
_lib = None


def lib():
    """Load the shared library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                                   "`python -m nvfp4_weight_quantized_gemv_gb300.buildlib`")
            L = ctypes.CDLL(LIB_PATH)
            vp, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            L.nvfp4_selftest_wait_timeout.argtypes = [vp]
            L.nvfp4_selftest_wait_timeout.restype = i
            L.nvfp4_gemv_batched.argtypes = [vp, vp, vp, vp, vp, i, i, i, vp]
            L.nvfp4_gemv_batched.restype = i
            L.nvfp4_gemv_batched_ex.argtypes = [vp, vp, vp, vp, vp, i, i, i, vp, ctypes.POINTER(nvfp4_gemv_opts)]
            L.nvfp4_gemv_batched_ex.restype = i
            L.nvfp4_gemv_batched_noalloc.argtypes = [vp, vp, vp, vp, vp, i, i, i, vp]
            L.nvfp4_gemv_batched_noalloc.restype = i
            L.nvfp4_gemv_swiglu.argtypes = [vp, vp, vp, vp, vp, i, i, i, vp]
            L.nvfp4_gemv_swiglu.restype = i
            L.nvfp4_ffn_swiglu.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, vp]
            L.nvfp4_ffn_swiglu.restype = i
            L.nvfp4_moe_gemv_grouped.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, vp]
            L.nvfp4_moe_gemv_grouped.restype = i
            L.nvfp4_gemv_workspace_size.argtypes = [i, i, i, ctypes.POINTER(nvfp4_gemv_opts), ctypes.POINTER(sz)]
            L.nvfp4_gemv_workspace_size.restype = i
            L.nvfp4_gemv_plan.argtypes = [i, i, i, ctypes.POINTER(nvfp4_gemv_opts),
                                          ctypes.POINTER(nvfp4_gemv_plan_info)]
            L.nvfp4_gemv_plan.restype = i
            L.nvfp4_quantize_ref.argtypes = [vp, i, i, vp, vp, vp]
            L.nvfp4_quantize_ref.restype = i
            L.nvfp4_quantize.argtypes = [vp, i, i, vp, vp, vp, vp]
            L.nvfp4_quantize.restype = i
            L.nvfp4_quantize_bf16.argtypes = [vp, i, i, vp, vp, vp, vp]
            L.nvfp4_quantize_bf16.restype = i
            L.nvfp4_device_error.argtypes = [vp, ctypes.POINTER(i)]
            L.nvfp4_device_error.restype = i
            L.nvfp4_last_error.argtypes = []
            L.nvfp4_last_error.restype = ctypes.c_char_p
            L.nvfp4_version.argtypes = []
            L.nvfp4_version.restype = i
            _lib = L
    return _lib


def nvfp4_last_error() -> str:
    return lib().nvfp4_last_error().decode()


def nvfp4_version() -> int:
    return lib().nvfp4_version()


def _check(status: int):
    if status != NVFP4_OK:
        raise Nvfp4Error(status, nvfp4_last_error())


def _opts(variant=0, tiling=0, num_ctas=0, stages=0, workspace=None, inflight=0):
    o = nvfp4_gemv_opts()
    o.variant, o.tiling, o.num_ctas, o.stages = int(variant), int(tiling), int(num_ctas), int(stages)
    o.inflight = int(inflight)
    if workspace is not None:
        o.workspace = workspace.data_ptr()
        o.workspace_bytes = workspace.numel() * workspace.element_size()
    return o


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _gemv_args(w_packed, w_scale, w_global_scale, x, y):
    import torch
    for name, t, dt in (("w_packed", w_packed, torch.uint8), ("w_scale", w_scale, torch.uint8),
                        ("w_global_scale", w_global_scale, torch.float32), ("y", y, torch.bfloat16)):
        if t.dtype != dt or not t.is_cuda or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous CUDA {dt} tensor")
    if x.dtype not in (torch.bfloat16,) or not x.is_cuda or not x.is_contiguous():
        raise TypeError("x must be a contiguous CUDA bfloat16 tensor")
    N = w_packed.shape[0]
    K = 2 * w_packed.shape[1]
    n = x.shape[0] if x.dim() == 2 else 1
    if w_scale.shape != (N, K // 16) or x.numel() != n * K or y.numel() != n * N:
        raise ValueError("shape mismatch: w_packed [N, K/2], w_scale [N, K/16], x [n, K], y [n, N]")
    return n, N, K


def nvfp4_gemv_batched(w_packed, w_scale, w_global_scale, x, y=None, stream=None):
    """Y[n, N] = X[n, K] . W^T (see include/nvfp4_gemv.h).  Returns y."""
    import torch
    if y is None:
        n = x.shape[0] if x.dim() == 2 else 1
        y = torch.empty((n, w_packed.shape[0]), dtype=torch.bfloat16, device=x.device)
    n, N, K = _gemv_args(w_packed, w_scale, w_global_scale, x, y)
    _check(lib().nvfp4_gemv_batched(w_packed.data_ptr(), w_scale.data_ptr(), w_global_scale.data_ptr(),
                                    x.data_ptr(), y.data_ptr(), n, N, K, _stream_handle(stream)))
    return y


def nvfp4_gemv_swiglu(w_packed, w_scale, w_global_scale, x, h=None, stream=None):
    """h[n, F] = bf16(silu(gate) * up) with gate/up rows interleaved in W [2F, K] (see the C header)."""
    import torch
    F = w_packed.shape[0] // 2
    n = x.shape[0] if x.dim() == 2 else 1
    K = x.shape[-1]
    if h is None:
        h = torch.empty((n, F), dtype=torch.bfloat16, device=x.device)
    _check(lib().nvfp4_gemv_swiglu(w_packed.data_ptr(), w_scale.data_ptr(), w_global_scale.data_ptr(), x.data_ptr(),
                                   h.data_ptr(), n, F, K, _stream_handle(stream)))
    return h


def nvfp4_ffn_swiglu(w_gu, w_down, x, h=None, y=None, stream=None):
    """Dense SwiGLU FFN: w_gu = (packed [2F, D/2], scale [2F, D/16], g [1]) with gate/up rows interleaved,
    w_down = (packed [D, F/2], scale [D, F/16], g [1]); x [n, D] bf16.  Returns y [n, D]."""
    import torch
    gp, gsc, gg = w_gu
    dp, dsc, dg = w_down
    n, D = x.shape
    F = gp.shape[0] // 2
    if h is None:
        h = torch.empty((n, F), dtype=torch.bfloat16, device=x.device)
    if y is None:
        y = torch.empty((n, D), dtype=torch.bfloat16, device=x.device)
    _check(lib().nvfp4_ffn_swiglu(gp.data_ptr(), gsc.data_ptr(), gg.data_ptr(), dp.data_ptr(), dsc.data_ptr(),
                                  dg.data_ptr(), x.data_ptr(), h.data_ptr(), y.data_ptr(), n, D, F,
                                  _stream_handle(stream)))
    return y


def nvfp4_moe_gemv_grouped(w_packed, w_scale, w_global_scale, x, expert_offsets, sorted_token, y=None,
                           swiglu=False, stream=None):
    """Grouped read-once GEMV over routed experts (see the C header).

    w_packed uint8 [E, N, K/2], w_scale uint8 [E, N, K/16], w_global_scale float32 [E], x bf16 [n, K],
    expert_offsets int32 [E+1], sorted_token int32 [A].  Returns y bf16 [A, N] (swiglu: [A, N/2])."""
    import torch
    E, N, half_k = w_packed.shape
    K = 2 * half_k
    A = sorted_token.numel()
    if y is None:
        y = torch.empty((A, N // 2 if swiglu else N), dtype=torch.bfloat16, device=x.device)
    _check(lib().nvfp4_moe_gemv_grouped(w_packed.data_ptr(), w_scale.data_ptr(), w_global_scale.data_ptr(),
                                        x.data_ptr(), expert_offsets.data_ptr(), sorted_token.data_ptr(),
                                        y.data_ptr(), E, A, x.shape[0], N, K, int(bool(swiglu)),
                                        _stream_handle(stream)))
    return y


def nvfp4_gemv_batched_ex(w_packed, w_scale, w_global_scale, x, y=None, stream=None, variant=0, tiling=0,
                          num_ctas=0, stages=0, workspace=None, inflight=0):
    """nvfp4_gemv_batched with explicit variant / tiling / grid / ring depth / workspace / stages in flight."""
    import torch
    if y is None:
        n = x.shape[0] if x.dim() == 2 else 1
        y = torch.empty((n, w_packed.shape[0]), dtype=torch.bfloat16, device=x.device)
    n, N, K = _gemv_args(w_packed, w_scale, w_global_scale, x, y)
    o = _opts(variant, tiling, num_ctas, stages, workspace, inflight)
    _check(lib().nvfp4_gemv_batched_ex(w_packed.data_ptr(), w_scale.data_ptr(), w_global_scale.data_ptr(),
                                       x.data_ptr(), y.data_ptr(), n, N, K, _stream_handle(stream),
                                       ctypes.byref(o)))
    return y


def nvfp4_gemv_batched_noalloc(w_packed, w_scale, w_global_scale, x, y, stream=None):
    """Allocation-free variant for callers that cannot call cudaMalloc (see the C header).

    `y` must be provided by the caller; the library allocates nothing.  Calls
    that can overlap on the GPU share one scratch array and race."""
    n, N, K = _gemv_args(w_packed, w_scale, w_global_scale, x, y)
    _check(lib().nvfp4_gemv_batched_noalloc(w_packed.data_ptr(), w_scale.data_ptr(), w_global_scale.data_ptr(),
                                            x.data_ptr(), y.data_ptr(), n, N, K, _stream_handle(stream)))
    return y


def nvfp4_gemv_workspace_size(n, N, K, variant=0, tiling=0, num_ctas=0, stages=0) -> int:
    b = ctypes.c_size_t(0)
    o = _opts(variant, tiling, num_ctas, stages)
    _check(lib().nvfp4_gemv_workspace_size(n, N, K, ctypes.byref(o), ctypes.byref(b)))
    return b.value


def nvfp4_gemv_plan(n, N, K, variant=0, tiling=0, num_ctas=0, stages=0, workspace_bytes=0) -> dict:
    info = nvfp4_gemv_plan_info()
    o = _opts(variant, tiling, num_ctas, stages)
    o.workspace_bytes = int(workspace_bytes)  # a declared scratch size caps the plan
    _check(lib().nvfp4_gemv_plan(n, N, K, ctypes.byref(o), ctypes.byref(info)))
    return dict(variant=VARIANT_NAMES[info.variant], tiling=TILING_NAMES[info.tiling], passes=info.passes,
                tile_tokens=list(info.tile_tokens[:min(info.passes, 16)]), num_ctas=info.num_ctas,
                stages=info.stages, smem_bytes=info.smem_bytes, units=info.units)


def nvfp4_quantize_ref(w):
    """Host quantizer: fp32 numpy W[N, K] -> (packed uint8 [N, K/2], scale uint8 [N, K/16], g float)."""
    import numpy as np
    w = np.ascontiguousarray(w, dtype=np.float32)
    N, K = w.shape
    packed = np.empty((N, K // 2), dtype=np.uint8)
    scale = np.empty((N, K // 16), dtype=np.uint8)
    g = np.zeros(1, dtype=np.float32)
    _check(lib().nvfp4_quantize_ref(w.ctypes.data, N, K, packed.ctypes.data, scale.ctypes.data, g.ctypes.data))
    return packed, scale, float(g[0])


def _quantize_into(w, packed, scale, g, stream=None):
    import torch
    if w.dim() != 2 or not w.is_cuda or not w.is_contiguous():
        raise ValueError("w must be a contiguous 2-D CUDA tensor")
    N, K = w.shape
    if w.dtype == torch.float32:
        fn = lib().nvfp4_quantize
    elif w.dtype == torch.bfloat16:
        fn = lib().nvfp4_quantize_bf16
    else:
        raise ValueError(f"w must be float32 or bfloat16, not {w.dtype}")
    _check(fn(w.data_ptr(), N, K, packed.data_ptr(), scale.data_ptr(), g.data_ptr(), _stream_handle(stream)))


def nvfp4_quantize(w, stream=None):
    """Device quantizer: CUDA float32 or bfloat16 W[N, K] -> (packed uint8 [N, K/2],
    scale uint8 [N, K/16], g float32 [1]), all on W's device, written asynchronously
    on `stream`.  Dispatches to nvfp4_quantize / nvfp4_quantize_bf16 by dtype."""
    import torch
    N, K = w.shape
    packed = torch.empty((N, K // 2), dtype=torch.uint8, device=w.device)
    scale = torch.empty((N, K // 16), dtype=torch.uint8, device=w.device)
    g = torch.empty(1, dtype=torch.float32, device=w.device)
    _quantize_into(w, packed, scale, g, stream)
    return packed, scale, g


def nvfp4_quantize_bf16(w, stream=None):
    """nvfp4_quantize for a bfloat16 W only (raises for any other dtype)."""
    import torch
    if w.dtype != torch.bfloat16:
        raise ValueError(f"nvfp4_quantize_bf16 takes bfloat16 weights, not {w.dtype}")
    return nvfp4_quantize(w, stream)


def nvfp4_device_error(stream=None) -> int:
    """Synchronize, read and clear the device error word.  Returns the word
    (0 = none; bits 8, 16 and 32 flag inputs a kernel could not use, bit 128 a
    failed index check of the debug-bounds build) and raises Nvfp4Error when a
    kernel gave up on a wait (bits 1, 2, 4)."""
    code = ctypes.c_int(0)
    st = lib().nvfp4_device_error(_stream_handle(stream), ctypes.byref(code))
    if st not in (NVFP4_OK, NVFP4_ERR_DEVICE_TIMEOUT, NVFP4_ERR_DEVICE_INPUT, NVFP4_ERR_DEVICE_BOUNDS):
        _check(st)
    if st == NVFP4_ERR_DEVICE_TIMEOUT:
        raise Nvfp4Error(st, nvfp4_last_error())
    return code.value


def nvfp4_selftest_wait_timeout(stream=None) -> None:
    """Enqueue the bounded-wait self-test kernel (a wait that nothing ends; it
    gives up after about 2 s and sets the device error word's timeout bit)."""
    _check(lib().nvfp4_selftest_wait_timeout(_stream_handle(stream)))


def build(force: bool = False) -> str:
    from .buildlib import build as _build
    return _build(force=force)
