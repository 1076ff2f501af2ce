"""fa_bwd_static_workspace: the backward pass for callers that cannot allocate.

Some callers cannot call cudaMalloc where they run the backward pass (a
framework that owns all device memory, a plugin that may not allocate behind
its host, code that must not synchronise on an allocation).  For them the
library offers fa_bwd_static_workspace, which keeps the backward pass's
scratch in a fixed 16 MiB array inside the library instead of a workspace the
caller allocates.

These tests call it through the C ABI.  Before each checked call the array is
filled with another problem's scratch (a call on different inputs), so a
value the checked call failed to write would show.  The result must equal, bit
for bit, fa_bwd given a caller-allocated workspace of the array's size (the
backward pass is deterministic and picks its kernels by the workspace it is
given), and must match the fp64 oracle.

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


def _device_case(case, seed, dout_scale=1.0):
    B, Hq, Hkv, N, d, causal, window, lengths = case
    x = make_case(B, Hq, Hkv, N, d, seed=seed, lengths=lengths)
    q, k, v, do = (to_dev(x[n]) for n in ("q", "k", "v", "dout"))
    if dout_scale != 1.0:
        do = (do.float() * dout_scale).to(do.dtype)
    return x, q, k, v, do


@pytest.mark.parametrize("case", CASES, ids=["dense_d128", "packed_d64_window"])
def test_static_workspace_matches_fa_bwd_bitwise(fa, oracle_mod, case):
    import torch
    B, Hq, Hkv, N, d, causal, window, lengths = case
    T = int(sum(lengths)) if lengths else 0
    scale = scale_of(d)
    stream = torch.cuda.current_stream()

    def run_static(q, k, v, o, lse, do, cu):
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        fa.fa_bwd_static_workspace(q, k, v, o, lse, do, dq, dk, dv, B, Hq, Hkv, N, d, causal,
                                   window, cu, T, scale, stream)
        fa.fa_device_status(stream)
        return dq, dk, dv

    x, q, k, v, do = _device_case(case, seed=21)
    cu = cu_dev(x["cu"])
    kw = dict(causal=causal, window=window, scale=scale, cu_seqlens=cu, max_seqlen=N)
    o, lse = fa.attention_forward(q, k, v, **kw)
    # fa_bwd with a caller-allocated workspace of the static array's size
    ws = torch.empty(fa.FA_STATIC_WORKSPACE_BYTES, dtype=torch.uint8, device=q.device)
    ref = fa.attention_backward(q, k, v, o, lse, do, workspace=ws, **kw)
    torch.cuda.synchronize()

    # another problem of the same shape (other inputs, larger dO) to fill the array
    _, q2, k2, v2, do2 = _device_case(case, seed=77, dout_scale=3.0)
    o2, lse2 = fa.attention_forward(q2, k2, v2, **kw)

    for _ in range(2):
        run_static(q2, k2, v2, o2, lse2, do2, cu)        # leaves its own scratch in the array
        got = run_static(q, k, v, o, lse, do, cu)
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            assert torch.equal(g.view(torch.int16), r.view(torch.int16)), name

    rq, rk, rv = oracle_mod.attention_bwd(x["q"], x["k"], x["v"], x["dout"], causal=causal,
                                          window=window, scale=scale, cu_seqlens=x["cu"])
    for name, g, r in (("dq", got[0], rq), ("dk", got[1], rk), ("dv", got[2], rv)):
        err = rel_fro(to_f64(g), r)
        assert err <= GRAD_REL_FRO, (name, err)


def test_static_workspace_rejects_sizes_beyond_its_array(fa):
    import exact_io_aware_tcgen05_gb300 as pkg
    # B * Hq * N = 4 * 64 * 32768 fp32 row statistics = 32 MiB > 16 MiB: rejected before
    # anything touches the GPU (the pointers are never dereferenced)
    assert pkg.fa_bwd_workspace_size(4, 64, 8, 32768, 128, 0) > pkg.FA_STATIC_WORKSPACE_BYTES
    st = pkg.fa_bwd_static_workspace(16, 16, 16, 16, 16, 16, 16, 16, 16, 4, 64, 8, 32768, 128,
                                     1, 0, None, 0, 0.1, None, check=False)
    assert st == pkg.FA_ERR_WORKSPACE
    assert "static array" in pkg.fa_last_error()
