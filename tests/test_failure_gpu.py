"""Failure detection without a GPU fault: every wait inside the kernels is bounded.

Setting the wait budget to one cycle makes every wait that is not already
satisfied give up.  The kernels must then abort cleanly (drain their own copies
and MMAs, free TMEM, exit), report FA_ERR_TIMEOUT through fa_device_status, and
leave the context usable: the next call with the default budget must be correct.
"""
import numpy as np
import pytest

from helpers import GRAD_REL_FRO, O_MAX_ABS, make_case, max_abs, rel_fro, scale_of, to_dev, to_f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("path,d", [("split", 128), ("fused", 128), ("fused", 64)])
def test_wait_budget_expiry_reports_timeout_then_recovers(fa, oracle_mod, path, d):
    import torch
    B, Hq, Hkv, N = 2, 4, 2, 700
    x = make_case(B, Hq, Hkv, N, d, seed=13)
    q, k, v, do = (to_dev(x[n]) for n in ("q", "k", "v", "dout"))
    stream = torch.cuda.current_stream()
    kw = dict(causal=True, scale=scale_of(d))
    fa.fa_device_status(stream)                     # start from a clean status word
    fa.fa_set_wait_limit_cycles(1)
    try:
        o, lse = fa.attention_forward(q, k, v, **kw)
        assert fa.fa_device_status(stream, check=False) == fa.FA_ERR_TIMEOUT
        fa.attention_backward(q, k, v, o, lse, do, path=path, **kw)
        assert fa.fa_device_status(stream, check=False) == fa.FA_ERR_TIMEOUT
    finally:
        fa.fa_set_wait_limit_cycles(0)              # back to the default budget
    assert fa.fa_device_status(stream, check=False) == fa.FA_OK
    o, lse = fa.attention_forward(q, k, v, **kw)
    dq, dk, dv = fa.attention_backward(q, k, v, o, lse, do, path=path, **kw)
    fa.fa_device_status(stream)
    o_ref, _ = oracle_mod.attention_fwd(x["q"], x["k"], x["v"], causal=True, scale=scale_of(d))
    assert max_abs(to_f64(o), o_ref) <= O_MAX_ABS
    refs = oracle_mod.attention_bwd(x["q"], x["k"], x["v"], x["dout"], causal=True,
                                    scale=scale_of(d))
    for g, r in zip((dq, dk, dv), refs):
        assert rel_fro(to_f64(g), r) <= GRAD_REL_FRO
