"""Shared helpers of the GPU tests: the tolerance, the oracle comparisons and
the device copies of the seeded inputs."""
import math

import numpy as np
import torch

import workloads
from oracle import attention as A

# Parity bar for bf16 results against the fp64 oracle: normalised L2 error and
# max absolute error (per output tensor).
REL_TOL = 5e-3
ABS_TOL = 2e-2
LSE_ABS_TOL = 1e-3


def err(x, ref):
    x = x.double().cpu().numpy() if isinstance(x, torch.Tensor) else np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-30)), float(np.abs(x - ref).max())


def assert_close(name, x, ref, rel=REL_TOL, abs_=ABS_TOL):
    if not np.any(np.asarray(ref)):
        # exactly-zero reference (e.g. dQ with one key): the relative error is
        # undefined; the result must be zero up to fp32 cancellation noise
        m = err(x, ref)[1]
        assert m <= 1e-6, f"{name}: reference is exactly 0, max abs {m:.3e} (<= 1e-6)"
        return
    r, m = err(x, ref)
    assert r <= rel and m <= abs_, f"{name}: rel {r:.3e} (<= {rel}), max abs {m:.3e} (<= {abs_})"


class Problem:
    """Seeded inputs on the host (bf16 and exact fp64 copies) and on cuda:0."""

    def __init__(self, B, H, S, D, causal, gain=1.0, seed=workloads.SEED):
        self.B, self.H, self.S, self.D, self.causal = B, H, S, D, causal
        self.scale = 1.0 / math.sqrt(D)
        self.host = workloads.make_inputs(B, H, S, D, gain, seed)
        self.f64 = [t.double().numpy() for t in self.host]
        dev = torch.device("cuda:0")
        self.q, self.k, self.v, self.do = (t.to(dev) for t in self.host)

    def oracle_fwd(self, heads=None):
        q, k, v, _ = self.f64
        if heads is None:
            return A.forward(q, k, v, self.causal, self.scale)
        return A.forward_heads(q, k, v, self.causal, self.scale, heads)
