"""Backward pass on the GPU (through the C ABI) against the fp64 oracle."""
import numpy as np
import pytest

from helpers import (GRAD_REL_FRO, cu_dev, make_case, rel_fro, scale_of, to_dev, to_f64)

pytestmark = pytest.mark.gpu

# (B, Hq, Hkv, N, d, causal, window, lengths)
SMALL = [
    (1, 1, 1, 128, 64, False, 0, None),
    (2, 4, 2, 300, 128, False, 0, None),       # ragged tail, GQA 2:1
    (2, 4, 2, 300, 128, True, 0, None),
    (1, 2, 2, 513, 64, True, 0, None),
    (1, 8, 1, 700, 128, True, 200, None),      # MQA + sliding window
    (1, 4, 4, 1000, 64, True, 129, None),
    (1, 2, 1, 1, 128, True, 0, None),          # a single token
    (6, 4, 2, 513, 128, True, 0, (1, 127, 128, 129, 300, 513)),   # packed batch
    (6, 4, 2, 513, 64, True, 0, (1, 127, 128, 129, 300, 513)),
    (3, 2, 1, 900, 128, False, 0, (900, 5, 256)),
    (4, 4, 1, 700, 128, True, 100, (700, 33, 256, 1)),
    # the backward's work order takes heads in chunks of 8: 18 query-head pairs (dQ:
    # 8 + 8 + 2) and 9 key/value-head pairs (dK/dV: 8 + 1); packed, 12 query heads
    # per sequence (8 + 4)
    (3, 6, 3, 300, 128, True, 0, None),
    (2, 12, 4, 300, 64, True, 0, (300, 77)),
    # degenerate masks: a window of one key (each query sees only itself), a window
    # wider than the sequence (plain causal), and a packed batch of 1- to 3-token
    # sequences
    (1, 2, 1, 300, 64, True, 1, None),
    (2, 2, 2, 260, 128, True, 5000, None),
    (5, 2, 1, 3, 64, True, 0, (1, 2, 3, 1, 1)),
    # empty sequences in a packed batch (no work items; the others unaffected)
    (4, 4, 2, 130, 64, True, 0, (5, 0, 130, 0)),
]


def run_fwd_bwd(fa, x, N, d, causal, window):
    import torch
    q, k, v, do = (to_dev(x[n]) for n in ("q", "k", "v", "dout"))
    cu = cu_dev(x["cu"])
    kw = dict(causal=causal, window=window, scale=scale_of(d), cu_seqlens=cu, max_seqlen=N)
    o, lse = fa.attention_forward(q, k, v, **kw)
    dq, dk, dv = fa.attention_backward(q, k, v, o, lse, do, **kw)
    fa.fa_device_status(torch.cuda.current_stream())
    return dq, dk, dv


@pytest.mark.parametrize("case", SMALL, ids=lambda c: f"B{c[0]}h{c[1]}x{c[2]}n{c[3]}d{c[4]}c{int(c[5])}w{c[6]}{'p' if c[7] else ''}")
def test_backward_matches_oracle(fa, oracle_mod, case):
    B, Hq, Hkv, N, d, causal, window, lengths = case
    x = make_case(B, Hq, Hkv, N, d, seed=5, lengths=lengths)
    dq, dk, dv = run_fwd_bwd(fa, x, N, d, causal, window)
    rq, rk, rv = oracle_mod.attention_bwd(x["q"], x["k"], x["v"], x["dout"], causal=causal,
                                          window=window, scale=scale_of(d), cu_seqlens=x["cu"])
    for name, g, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        err = rel_fro(to_f64(g), ref)
        assert err <= GRAD_REL_FRO, (name, err)


@pytest.mark.parametrize("case", [(1, 8, 2, 1100, 128, None), (3, 8, 2, 1100, 64, (1100, 7, 640))],
                         ids=["d128", "d64packed"])
def test_backward_is_deterministic(fa, case):
    """Two runs give the same bits: every gradient row is summed by one CTA in a
    fixed order (both head dimensions; their rings and warpgroups differ)."""
    import torch
    B, Hq, Hkv, N, d, lengths = case
    x = make_case(B, Hq, Hkv, N, d, seed=9, lengths=lengths)
    a = run_fwd_bwd(fa, x, N, d, True, 0)
    b = run_fwd_bwd(fa, x, N, d, True, 0)
    for ga, gb in zip(a, b):
        assert torch.equal(ga.view(torch.int16), gb.view(torch.int16))
