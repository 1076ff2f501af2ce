"""fa_bwd_static_workspace: the backward pass for callers that cannot allocate.

Some callers cannot call cudaMalloc where they run the backward pass (a
framework that owns all device memory, a plugin that may not allocate behind
its host, code that must not synchronise on an allocation).  For them the
library offers fa_bwd_static_workspace, which keeps the backward pass's
scratch in a fixed 16 MiB array inside the library instead of a workspace the
caller allocates.  These tests call it through the C ABI and check it against
fa_bwd with a caller-allocated workspace, twice in a row (the array keeps the
previous call's contents, which must not matter).

This file is collected last on purpose: it must pass on its own in a fresh
process and after every other test.
"""
import pytest

from helpers import GRAD_REL_FRO, cu_dev, make_case, rel_fro, scale_of, to_dev, to_f64

pytestmark = pytest.mark.gpu

CASES = [
    # (B, Hq, Hkv, N, d, causal, window, lengths)
    (2, 4, 2, 300, 128, True, 0, None),
    (4, 4, 1, 700, 64, True, 100, (700, 33, 256, 1)),
]


@pytest.mark.parametrize("case", CASES, ids=["dense_d128", "packed_d64_window"])
def test_static_workspace_matches_fa_bwd_twice(fa, case):
    import torch
    B, Hq, Hkv, N, d, causal, window, lengths = case
    x = make_case(B, Hq, Hkv, N, d, seed=21, lengths=lengths)
    q, k, v, do = (to_dev(x[n]) for n in ("q", "k", "v", "dout"))
    cu = cu_dev(x["cu"])
    T = int(sum(lengths)) if lengths else 0
    kw = dict(causal=causal, window=window, scale=scale_of(d), cu_seqlens=cu, max_seqlen=N)
    o, lse = fa.attention_forward(q, k, v, **kw)
    ref = fa.attention_backward(q, k, v, o, lse, do, **kw)     # caller-allocated workspace
    stream = torch.cuda.current_stream()
    for _ in range(2):
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        fa.fa_bwd_static_workspace(q, k, v, o, lse, do, dq, dk, dv, B, Hq, Hkv, N, d, causal,
                                   window, cu, T, scale_of(d), stream)
        fa.fa_device_status(stream)
        for g, r in zip((dq, dk, dv), ref):
            assert rel_fro(to_f64(g), to_f64(r)) <= GRAD_REL_FRO


def test_static_workspace_rejects_sizes_beyond_its_array(fa):
    import exact_io_aware_tcgen05_gb300 as pkg
    # B * Hq * N = 4 * 64 * 32768 fp32 row statistics = 32 MiB > 16 MiB: rejected before
    # anything touches the GPU (the pointers are never dereferenced)
    assert pkg.fa_bwd_workspace_size(4, 64, 8, 32768, 128, 0) > 16 * 1024 * 1024
    st = pkg.fa_bwd_static_workspace(16, 16, 16, 16, 16, 16, 16, 16, 16, 4, 64, 8, 32768, 128,
                                     1, 0, None, 0, 0.1, None, check=False)
    assert st == pkg.FA_ERR_WORKSPACE
    assert "static array" in pkg.fa_last_error()
