"""Helpers shared by the GPU parity tests (comparison metrics, tolerances)."""
import numpy as np
import torch

# max |gpu - oracle| / RMS(oracle), per output tensor: the bar for fp32 inputs
# and for bf16 inputs.
TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def rel_err(gpu, ref):
    g = f64(gpu) if isinstance(gpu, torch.Tensor) else np.asarray(gpu, np.float64)
    r = np.asarray(ref, np.float64)
    rms = np.sqrt(np.mean(r * r))
    if rms == 0:
        return float(np.abs(g - r).max(initial=0.0))
    return float(np.abs(g - r).max(initial=0.0) / rms)


def assert_close(gpu, ref, dtype, what=""):
    e = rel_err(gpu, ref)
    assert e <= TOL[dtype], "%s: max|err|/RMS = %.3e > %.1e" % (what, e, TOL[dtype])
    return e


def canary_fill(t):
    """Fill a float tensor with a recognisable bit pattern (NaN-free)."""
    t.view(torch.int32).fill_(0x3E9E0F3C)    # ~0.3087
    return t
