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
    # without a causal mask at d = 64 (the default there is the fused backward)
    (2, 4, 2, 300, 64, False, 0, None),
    (4, 4, 1, 700, 64, False, 0, (700, 33, 256, 1)),
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


# the two backward paths: "fused" (the full workspace: one kernel, dQ summed across
# CTAs as int32 fixed point) and "split" (the least workspace: a dK/dV kernel and a dQ
# kernel)
PATHS = ["fused", "split"]


def run_fwd_bwd(fa, x, N, d, causal, window, path="fused"):
    import torch
    q, k, v, do = (to_dev(x[n]) for n in ("q", "k", "v", "dout"))
    cu = cu_dev(x["cu"])
    kw = dict(causal=causal, window=window, scale=scale_of(d), cu_seqlens=cu, max_seqlen=N)
    o, lse = fa.attention_forward(q, k, v, **kw)
    dq, dk, dv = fa.attention_backward(q, k, v, o, lse, do, path=path, **kw)
    fa.fa_device_status(torch.cuda.current_stream())
    return dq, dk, dv


def expected_path(fa, case, path):
    B, Hq, Hkv, N, d, causal, window, lengths = case
    T = int(sum(lengths)) if lengths else 0
    size = (fa.fa_bwd_workspace_size_min if path == "split" else fa.fa_bwd_workspace_size_fused)(
        B, Hq, Hkv, N, d, T)
    fa.fa_bwd_set_path(fa.FA_BWD_SPLIT if path == "split" else fa.FA_BWD_FUSED)
    try:
        return fa.fa_bwd_path(B, Hq, Hkv, N, d, causal, window, T, size)
    finally:
        fa.fa_bwd_set_path(fa.FA_BWD_AUTO)


_ORACLE = {}


def oracle_grads(oracle_mod, x, case):
    key = tuple(map(str, case))
    if key not in _ORACLE:
        B, Hq, Hkv, N, d, causal, window, lengths = case
        _ORACLE[key] = oracle_mod.attention_bwd(x["q"], x["k"], x["v"], x["dout"], causal=causal,
                                                window=window, scale=scale_of(d),
                                                cu_seqlens=x["cu"])
    return _ORACLE[key]


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("case", SMALL, ids=lambda c: f"B{c[0]}h{c[1]}x{c[2]}n{c[3]}d{c[4]}c{int(c[5])}w{c[6]}{'p' if c[7] else ''}")
def test_backward_matches_oracle(fa, oracle_mod, case, path):
    B, Hq, Hkv, N, d, causal, window, lengths = case
    assert expected_path(fa, case, path) == (fa.FA_BWD_FUSED if path == "fused" else fa.FA_BWD_SPLIT)
    x = make_case(B, Hq, Hkv, N, d, seed=5, lengths=lengths)
    dq, dk, dv = run_fwd_bwd(fa, x, N, d, causal, window, path)
    rq, rk, rv = oracle_grads(oracle_mod, x, case)
    for name, g, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        err = rel_fro(to_f64(g), ref)
        assert err <= GRAD_REL_FRO, (name, err)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("case", [(1, 8, 2, 1100, 128, True, None), (3, 8, 2, 1100, 64, True, (1100, 7, 640)),
                                  (2, 4, 2, 1100, 64, False, None)],
                         ids=["d128", "d64packed", "d64noncausal"])
def test_backward_is_deterministic(fa, case, path):
    """Two runs give the same bits.  Split: every gradient row is summed by one CTA in
    a fixed order.  Fused: dK and dV as in the split path; dQ is summed across CTAs
    as fixed-point integers, whose sum does not depend on the order of the additions
    (both head dimensions; their accumulator layouts differ)."""
    import torch
    B, Hq, Hkv, N, d, causal, lengths = case
    x = make_case(B, Hq, Hkv, N, d, seed=9, lengths=lengths)
    a = run_fwd_bwd(fa, x, N, d, causal, 0, path)
    b = run_fwd_bwd(fa, x, N, d, causal, 0, path)
    for ga, gb in zip(a, b):
        assert torch.equal(ga.view(torch.int16), gb.view(torch.int16))


@pytest.mark.parametrize("case", [
    (2, 16, 2, 1500, 128, True, 0, None),          # GQA 8:1, 12 key tiles: chains of up to 12
    (1, 4, 4, 2100, 64, True, 300, None),          # window: chains of 4 over 17 tiles
    (5, 8, 4, 900, 128, True, 0, (900, 1, 385, 0, 640)),   # packed, unaligned starts, empty
    (1, 8, 2, 2100, 64, False, 0, None),          # no mask: every row gets all 17 tiles
], ids=["gqa8_chain12", "d64_window300", "packed_mixed", "d64_noncausal17"])
def test_fused_backward_longer_chains(fa, oracle_mod, case):
    """The fused backward on cases whose dQ rows collect many contributions (long
    causal chains, a window, GQA 8:1, a packed batch with unaligned starts and an
    empty sequence, no mask over 17 key tiles), against the oracle."""
    B, Hq, Hkv, N, d, causal, window, lengths = case
    assert expected_path(fa, case, "fused") == fa.FA_BWD_FUSED
    x = make_case(B, Hq, Hkv, N, d, seed=17, lengths=lengths)
    dq, dk, dv = run_fwd_bwd(fa, x, N, d, causal, window, "fused")
    rq, rk, rv = oracle_grads(oracle_mod, x, case)
    for name, g, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        err = rel_fro(to_f64(g), ref)
        assert err <= GRAD_REL_FRO, (name, err)


def _many_lengths():
    """1100 packed sequences: seeded lengths in [0, 300) with empty, one-token and
    tile-edge lengths mixed in."""
    rng = np.random.default_rng(11)
    lengths = rng.integers(0, 300, size=1100)
    lengths[::97] = 0
    lengths[1::89] = 1
    lengths[2::83] = 128
    lengths[3::79] = 129
    return tuple(int(x) for x in lengths)


@pytest.mark.parametrize("d", [64, 128])
def test_many_packed_sequences(fa, oracle_mod, d):
    """More than a thousand packed sequences (the CTAs find their sequence by a
    binary search over cu_seqlens): forward element by element, and both backward
    paths, against the oracle."""
    from helpers import LSE_MAX_ABS, O_MAX_ABS, max_abs
    lengths = _many_lengths()
    B, Hq, Hkv, N = len(lengths), 2, 1, max(lengths)
    x = make_case(B, Hq, Hkv, N, d, seed=23, lengths=lengths)
    q, k, v, do = (to_dev(x[n]) for n in ("q", "k", "v", "dout"))
    cu = cu_dev(x["cu"])
    kw = dict(causal=True, window=0, scale=scale_of(d), cu_seqlens=cu, max_seqlen=N)
    o, lse = fa.attention_forward(q, k, v, **kw)
    o_ref, lse_ref = oracle_mod.attention_fwd(x["q"], x["k"], x["v"], causal=True,
                                              scale=scale_of(d), cu_seqlens=x["cu"])
    assert max_abs(to_f64(o), o_ref) <= O_MAX_ABS
    assert max_abs(lse.cpu().numpy().astype(np.float64), lse_ref) <= LSE_MAX_ABS
    refs = oracle_mod.attention_bwd(x["q"], x["k"], x["v"], x["dout"], causal=True,
                                    scale=scale_of(d), cu_seqlens=x["cu"])
    for path in PATHS:
        grads = fa.attention_backward(q, k, v, o, lse, do, path=path, **kw)
        fa.fa_device_status()
        for name, g, r in zip(("dq", "dk", "dv"), grads, refs):
            err = rel_fro(to_f64(g), r)
            assert err <= GRAD_REL_FRO, (path, name, err)


# The split backward's dQ CTA may serve several query heads of one key/value group
# (fa_bwd_set_dq_heads; the library's own choice gives more than one only on large
# grids).  Every divisor of the group must give the same bits, and they must match the
# oracle.  (B, Hq, Hkv, N, d, causal, window, lengths, dtype, dropout)
DQ_HEADS_CASES = [
    (2, 8, 2, 300, 128, True, 0, None, "bf16", None),
    (1, 8, 1, 700, 64, True, 200, None, "bf16", None),              # MQA, window
    (5, 4, 1, 513, 128, False, 0, (1, 127, 0, 129, 513), "f16", None),   # packed, empty seq
    (3, 6, 2, 260, 64, True, 0, (260, 1, 131), "bf16", None),        # group of 3
    (2, 4, 2, 384, 128, True, 0, None, "bf16", (0.1, 77, 3)),        # dropout: one head per CTA whatever is asked
    # 9 key tiles per head: Q, dO and the K/V tiles of up to 4 heads wrap the dQ kernel's
    # slot ring many times (items counted over all heads)
    (1, 8, 2, 1100, 64, False, 0, None, "bf16", None),
    (1, 8, 2, 1100, 128, True, 0, None, "bf16", None),
]


@pytest.mark.parametrize("case", DQ_HEADS_CASES,
                         ids=lambda c: f"B{c[0]}h{c[1]}x{c[2]}n{c[3]}d{c[4]}c{int(c[5])}w{c[6]}"
                                       f"{'p' if c[7] else ''}{c[8]}{'drop' if c[9] else ''}")
def test_dq_heads_per_cta_give_the_same_bits(fa, oracle_mod, case):
    import torch
    B, Hq, Hkv, N, d, causal, window, lengths, dtype, drop = case
    x = make_case(B, Hq, Hkv, N, d, seed=61, lengths=lengths, dtype=dtype)
    q, k, v, do = (to_dev(x[n]) for n in ("q", "k", "v", "dout"))
    kw = dict(causal=causal, window=window, scale=scale_of(d), cu_seqlens=cu_dev(x["cu"]),
              max_seqlen=N)
    o, lse = fa.attention_forward(q, k, v, dropout=drop, **kw)
    G = Hq // Hkv
    first = None
    for heads in [c for c in range(1, G + 1) if G % c == 0]:
        got = fa.attention_backward(q, k, v, o, lse, do, path="split", dq_heads=heads,
                                    dropout=drop, **kw)
        fa.fa_device_status(torch.cuda.current_stream())
        if first is None:
            first = got
            continue
        for name, a, b in zip(("dq", "dk", "dv"), got, first):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16)), (heads, name)
    if drop is None:
        refs = oracle_mod.attention_bwd(x["q"], x["k"], x["v"], x["dout"], causal=causal,
                                        window=window, scale=scale_of(d), cu_seqlens=x["cu"])
        for name, g, r in zip(("dq", "dk", "dv"), first, refs):
            assert rel_fro(to_f64(g), r) <= GRAD_REL_FRO, name
