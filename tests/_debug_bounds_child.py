"""Child process of tests/test_debug_bounds.py: the same GEMV calls through
the library built with -DNVFP4_DEBUG_BOUNDS (device checks of the computed
workspace indices).  Prints one JSON line per case: the worst error over the
tolerance against the oracle and the device error word."""
from __future__ import annotations

import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import nvfp4_weight_quantized_gemv_gb300 as nv  # noqa: E402
import oracle  # noqa: E402
import synth  # noqa: E402

nv.LIB_PATH = nv.DEBUG_LIB_PATH
from nvfp4_weight_quantized_gemv_gb300 import buildlib  # noqa: E402

buildlib.build(debug_bounds=True)
oracle.build()
assert nv.lib()._name == nv.DEBUG_LIB_PATH

# (variant, N, K, n, num_ctas): whole row blocks, row blocks summed in
# clusters, uneven splits through the workspace, stream-K, two token passes
CASES = [("fp4", 1024, 3072, 5, 0), ("fp4", 1024, 3072, 5, 24), ("fp4", 1024, 3072, 16, 40),
         ("fp4", 1000, 1024, 9, 0), ("fp4", 1024, 3072, 20, 38), ("tc", 1024, 3072, 5, 40),
         ("tc", 1000, 1024, 24, 0), ("mma", 1000, 1024, 5, 0), ("simt", 384, 2048, 3, 0)]
VARIANT = {"fp4": nv.VARIANT_FP4, "tc": nv.VARIANT_TC, "mma": nv.VARIANT_MMA, "simt": nv.VARIANT_SIMT}
for variant, N, K, n, ctas in CASES:
    packed, scale, g = oracle.quantize(synth.weights_f32(N, K, N + K))
    x = synth.activations_bf16(n, K, 3)
    y64, _ = oracle.gemv(packed, scale, g, x)
    wp = torch.from_numpy(packed).cuda()
    ws = torch.from_numpy(scale).cuda()
    gs = torch.tensor([g], dtype=torch.float32, device="cuda")
    xt = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    y = nv.nvfp4_gemv_batched_ex(wp, ws, gs, xt, variant=VARIANT[variant], num_ctas=ctas)
    torch.cuda.synchronize()
    word = nv.nvfp4_device_error()
    err = np.abs(y.double().cpu().numpy() - y64) / (1e-2 * (np.abs(y64) + 1.0))
    print(json.dumps({"case": [variant, N, K, n, ctas], "worst_over_tol": float(err.max()), "error_word": word}),
          flush=True)
