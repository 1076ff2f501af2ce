"""Shared test helpers: seeded inputs, device transfer, comparison metrics."""
from __future__ import annotations

import math

import numpy as np

from exact_io_aware_tcgen05_gb300.inputs import attention_inputs, cu_seqlens_of

# Tolerances: bf16 inputs from N(0, 1), fp32 accumulation, bf16 outputs.
O_MAX_ABS = 2e-2        # forward output, max abs error vs the fp64 oracle
LSE_MAX_ABS = 1e-3      # logsumexp (fp32), max abs error
GRAD_REL_FRO = 2e-2     # dQ, dK, dV: ||g - g*||_F / ||g*||_F


def make_case(B, Hq, Hkv, N, d, seed, lengths=None, with_dout=True, dtype="bf16"):
    """Seeded inputs in the dense ([B, N, H, d]) or packed ([T, H, d]) layout
    (bf16 bit patterns, or float16 arrays for dtype "f16")."""
    if lengths is not None:
        T = int(sum(lengths))
        qs, kvs = (T, Hq, d), (T, Hkv, d)
        cu = cu_seqlens_of(lengths)
    else:
        qs, kvs = (B, N, Hq, d), (B, N, Hkv, d)
        cu = None
    x = attention_inputs(qs, kvs, seed, with_dout=with_dout, dtype=dtype)
    x["cu"] = cu
    return x


def to_dev(a):
    """bf16 bit patterns (uint16) -> a bf16 CUDA tensor; float16 -> a float16 one."""
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        return torch.from_numpy(a).cuda()
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()


def cu_dev(cu):
    import torch
    return None if cu is None else torch.from_numpy(np.asarray(cu, np.int32)).cuda()


def to_f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def rel_fro(g, ref):
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(g - ref) / den) if den > 0 else float(np.linalg.norm(g))


def max_abs(a, b):
    finite = np.isfinite(b)
    if not finite.all():
        assert np.array_equal(np.isfinite(a), finite), "non-finite pattern differs"
        assert (a[~finite] == b[~finite]).all()
    return float(np.abs(a[finite] - b[finite]).max()) if finite.any() else 0.0


def scale_of(d):
    return 1.0 / math.sqrt(d)
