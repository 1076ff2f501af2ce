"""A seeded random sweep of problem shapes through the C ABI, forward and backward,
against the fp64 oracle.

Each case draws: the head dimension (64 or 128); key/value heads and a GQA group of
1, 2 or 4 query heads each; a dense batch or a packed one whose lengths mix empty,
one- and two-token and longer sequences; a causal mask or none, and under a causal
mask sometimes a sliding window (from one key to wider than the sequence); bf16 or fp16
operands.  The backward runs the library's default path and, under causal masks, the
fused path as well.  Tolerances are those of the other parity tests.  For a GQA group of
more than one head the forward and the split backward also run with the whole group per
CTA (fa_fwd_set_heads, fa_bwd_set_dq_heads), which must give the same bits.
"""
import numpy as np
import pytest

from helpers import (GRAD_REL_FRO, LSE_MAX_ABS, O_MAX_ABS, cu_dev, make_case, max_abs, rel_fro,
                     scale_of, to_dev, to_f64)

pytestmark = pytest.mark.gpu


def draw_cases(n, seed=2026):
    rng = np.random.default_rng(seed)
    cases = []
    for _ in range(n):
        d = int(rng.choice([64, 128]))
        hkv = int(rng.choice([1, 2]))
        hq = hkv * int(rng.choice([1, 2, 4]))
        causal = bool(rng.random() < 0.7)
        if rng.random() < 0.5:
            b = int(rng.integers(1, 7))
            pool = [0, 1, 2] + list(rng.integers(3, 640, size=6))
            lengths = tuple(int(rng.choice(pool)) for _ in range(b))
            if max(lengths) == 0:
                lengths = lengths[:-1] + (int(rng.integers(1, 640)),)
            n_max = max(lengths)
        else:
            b = int(rng.integers(1, 3))
            lengths = None
            n_max = int(rng.integers(1, 700))
        window = int(rng.integers(1, n_max + 64)) if causal and rng.random() < 0.3 else 0
        dtype = "f16" if rng.random() < 0.3 else "bf16"
        cases.append((b, hq, hkv, n_max, d, causal, window, lengths, dtype))
    return cases


CASES = draw_cases(64)


def _id(c):
    b, hq, hkv, n, d, causal, window, lengths, dtype = c
    return f"B{b}h{hq}x{hkv}n{n}d{d}c{int(causal)}w{window}{'p' if lengths else ''}{dtype}"


@pytest.mark.parametrize("idx", range(len(CASES)), ids=[_id(c) for c in CASES])
def test_random_shapes_match_oracle(fa, oracle_mod, idx):
    import torch
    b, hq, hkv, n, d, causal, window, lengths, dtype = CASES[idx]
    seed = 1000 + idx
    x = make_case(b, hq, hkv, n, d, seed=seed, lengths=lengths, dtype=dtype)
    q, k, v, do = (to_dev(x[m]) for m in ("q", "k", "v", "dout"))
    kw = dict(causal=causal, window=window, scale=scale_of(d), cu_seqlens=cu_dev(x["cu"]),
              max_seqlen=n)
    o, lse = fa.attention_forward(q, k, v, **kw)
    fa.fa_device_status(torch.cuda.current_stream())
    ref = dict(causal=causal, window=window, scale=scale_of(d), cu_seqlens=x["cu"])
    o_ref, lse_ref = oracle_mod.attention_fwd(x["q"], x["k"], x["v"], **ref)
    assert max_abs(to_f64(o), o_ref) <= O_MAX_ABS
    assert max_abs(lse.cpu().numpy().astype(np.float64), lse_ref) <= LSE_MAX_ABS
    grads = oracle_mod.attention_bwd(x["q"], x["k"], x["v"], x["dout"], **ref)
    for path in ("auto", "fused"):
        got = fa.attention_backward(q, k, v, o, lse, do, path=path, **kw)
        fa.fa_device_status(torch.cuda.current_stream())
        for name, g, r in zip(("dq", "dk", "dv"), got, grads):
            assert rel_fro(to_f64(g), r) <= GRAD_REL_FRO, (path, name)
    G = hq // hkv
    if G > 1:
        o2, lse2 = fa.attention_forward(q, k, v, heads=G, **kw)
        split = fa.attention_backward(q, k, v, o, lse, do, path="split", **kw)
        grouped = fa.attention_backward(q, k, v, o, lse, do, path="split", dq_heads=G, **kw)
        fa.fa_device_status(torch.cuda.current_stream())
        assert torch.equal(o2.view(torch.int16), o.view(torch.int16)) and torch.equal(lse2, lse)
        for name, a, b in zip(("dq", "dk", "dv"), grouped, split):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16)), name
