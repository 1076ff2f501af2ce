"""fp16 inputs (fa_fwd_typed / fa_bwd_typed with FA_DTYPE_F16) against the fp64 oracle.

The same kernels run with fp16 operands in the tcgen05 products and fp16 outputs; P and
dS are rounded to fp16 before their products.  The oracle sees the same fp16 values,
upcast exactly.  Tolerances are those of the bf16 path (fp16 carries three more mantissa
bits, so they hold with room to spare).
"""
import numpy as np
import pytest

from helpers import (GRAD_REL_FRO, LSE_MAX_ABS, O_MAX_ABS, cu_dev, make_case, max_abs, rel_fro,
                     scale_of, to_dev, to_f64)

pytestmark = pytest.mark.gpu

# (B, Hq, Hkv, N, d, causal, window, lengths)
CASES = [
    (1, 1, 1, 128, 64, False, 0, None),
    (2, 4, 2, 300, 128, True, 0, None),
    (1, 2, 2, 513, 64, True, 0, None),
    (1, 8, 1, 700, 128, True, 200, None),
    (6, 4, 2, 513, 128, True, 0, (1, 127, 128, 129, 300, 513)),
    (6, 4, 2, 513, 64, True, 0, (1, 127, 128, 129, 300, 513)),
    (3, 2, 1, 900, 128, False, 0, (900, 5, 256)),
]


def _ids(c):
    return f"B{c[0]}h{c[1]}x{c[2]}n{c[3]}d{c[4]}c{int(c[5])}w{c[6]}{'p' if c[7] else ''}"


def _run(fa, x, N, d, causal, window, backward):
    import torch
    q, k, v = to_dev(x["q"]), to_dev(x["k"]), to_dev(x["v"])
    cu = cu_dev(x["cu"])
    kw = dict(causal=causal, window=window, scale=scale_of(d), cu_seqlens=cu, max_seqlen=N)
    o, lse = fa.attention_forward(q, k, v, **kw)
    out = {"o": o, "lse": lse}
    if backward:
        out["dq"], out["dk"], out["dv"] = fa.attention_backward(q, k, v, o, lse, to_dev(x["dout"]), **kw)
    fa.fa_device_status(torch.cuda.current_stream())
    assert o.dtype == q.dtype
    return out


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_f16_forward_and_backward_match_oracle(fa, oracle_mod, case):
    B, Hq, Hkv, N, d, causal, window, lengths = case
    x = make_case(B, Hq, Hkv, N, d, seed=21, lengths=lengths, dtype="f16")
    got = _run(fa, x, N, d, causal, window, backward=True)
    import torch
    assert got["o"].dtype == torch.float16 and got["dq"].dtype == torch.float16
    kw = dict(causal=causal, window=window, scale=scale_of(d), cu_seqlens=x["cu"])
    o_ref, lse_ref = oracle_mod.attention_fwd(x["q"], x["k"], x["v"], **kw)
    assert max_abs(to_f64(got["o"]), o_ref) <= O_MAX_ABS
    assert max_abs(got["lse"].cpu().numpy().astype(np.float64), lse_ref) <= LSE_MAX_ABS
    refs = oracle_mod.attention_bwd(x["q"], x["k"], x["v"], x["dout"], **kw)
    for name, ref in zip(("dq", "dk", "dv"), refs):
        assert rel_fro(to_f64(got[name]), ref) <= GRAD_REL_FRO, name


def test_f16_is_more_accurate_than_bf16_on_the_same_draws(fa, oracle_mod):
    """The same float32 draws rounded to fp16 give a forward output closer to its
    oracle than the bf16 rounding gives to its own: the fp16 path really runs in
    fp16 (a bf16 product on fp16 bits would be far off)."""
    errs = {}
    for dtype in ("bf16", "f16"):
        x = make_case(2, 4, 2, 300, 128, seed=5, with_dout=False, dtype=dtype)
        got = _run(fa, x, 300, 128, True, 0, backward=False)
        o_ref, _ = oracle_mod.attention_fwd(x["q"], x["k"], x["v"], causal=True, window=0,
                                            scale=scale_of(128))
        errs[dtype] = max_abs(to_f64(got["o"]), o_ref)
    assert errs["f16"] < errs["bf16"] / 2, errs


def test_f16_backward_is_deterministic(fa):
    import torch
    x = make_case(2, 4, 2, 700, 128, seed=3, dtype="f16")
    a = _run(fa, x, 700, 128, True, 0, backward=True)
    b = _run(fa, x, 700, 128, True, 0, backward=True)
    for n in ("o", "dq", "dk", "dv"):
        assert torch.equal(a[n].view(torch.int16), b[n].view(torch.int16)), n
