"""Helpers shared by the GPU parity tests (comparison metrics, tolerances)."""
import numpy as np
import torch

# max |gpu - oracle| / RMS(oracle), per output tensor: the bar for fp32 inputs
# and for bf16 inputs.
TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}

# Half an ulp of the tensor's own storage type, relative to the value: the
# error of rounding an exact result into that type.  A bf16 output carries it
# unavoidably (rounding the fp64 oracle itself to bf16 already gives
# 3.2e-2 x RMS on the small varlen case, where max|o| is 12 x RMS), so the
# bound applies to the error beyond it.
HALF_ULP = {torch.float32: 2.0 ** -24, torch.bfloat16: 2.0 ** -8}


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def rel_err(gpu, ref, storage=torch.float32):
    """max over elements of (|gpu - ref| - half_ulp(storage) |ref|)^+ / RMS(ref)."""
    g = f64(gpu) if isinstance(gpu, torch.Tensor) else np.asarray(gpu, np.float64)
    r = np.asarray(ref, np.float64)
    if r.size == 0:
        return 0.0
    excess = np.maximum(np.abs(g - r) - HALF_ULP[storage] * np.abs(r), 0.0)
    rms = np.sqrt(np.mean(r * r))
    return float(excess.max() / rms) if rms > 0 else float(excess.max())


def assert_close(gpu, ref, dtype, what=""):
    storage = gpu.dtype if isinstance(gpu, torch.Tensor) else torch.float32
    e = rel_err(gpu, ref, storage)
    assert e <= TOL[dtype], "%s: max|err|/RMS beyond output rounding = %.3e > %.1e" % (
        what, e, TOL[dtype])
    return e


def canary_fill(t):
    """Fill a float tensor with a recognisable bit pattern (NaN-free)."""
    t.view(torch.int32).fill_(0x3E9E0F3C)    # ~0.3087
    return t
