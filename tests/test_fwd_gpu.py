"""Forward pass on the GPU (through the C ABI) against the fp64 oracle."""
import numpy as np
import pytest

from helpers import (LSE_MAX_ABS, O_MAX_ABS, cu_dev, make_case, max_abs, scale_of, to_dev, to_f64)

pytestmark = pytest.mark.gpu

# (B, Hq, Hkv, N, d, causal, window, lengths)
SMALL = [
    (1, 1, 1, 128, 64, False, 0, None),        # one tile
    (2, 4, 2, 300, 128, False, 0, None),       # two CTAs per head, ragged tail
    (2, 4, 2, 300, 128, True, 0, None),
    (1, 2, 2, 513, 64, True, 0, None),
    (1, 8, 1, 700, 128, True, 200, None),      # MQA + sliding window
    (1, 4, 4, 1000, 64, True, 129, None),
    (1, 2, 1, 1, 128, True, 0, None),          # a single token
    (1, 2, 2, 1, 64, False, 0, None),
    (6, 4, 2, 513, 128, True, 0, (1, 127, 128, 129, 300, 513)),   # packed batch
    (6, 4, 2, 513, 64, True, 0, (1, 127, 128, 129, 300, 513)),
    (3, 2, 1, 900, 128, False, 0, (900, 5, 256)),
    (4, 4, 1, 700, 128, True, 100, (700, 33, 256, 1)),
    # 2 MB of K and V per head: the work order takes heads in chunks of 8, so 10
    # (sequence, head) pairs make a full chunk and a partial one; packed, 12 query
    # heads per sequence do the same within each sequence
    (1, 10, 5, 4096, 128, True, 0, None),
    (2, 12, 4, 4096, 128, True, 0, (4096, 300)),
    # 1 MB per head: chunks of 16, so 20 pairs make 16 + 4
    (2, 10, 10, 2048, 128, True, 0, None),
    # degenerate masks: a window of one key (each query sees only itself), a window
    # wider than the sequence (plain causal), and a packed batch of 1- to 3-token
    # sequences
    (1, 2, 1, 300, 64, True, 1, None),
    (2, 2, 2, 260, 128, True, 5000, None),
    (5, 2, 1, 3, 64, True, 0, (1, 2, 3, 1, 1)),
    # empty sequences in a packed batch (no work items; the others unaffected)
    (4, 4, 2, 130, 64, True, 0, (5, 0, 130, 0)),
]


def run_fwd(fa, x, B, Hq, Hkv, N, d, causal, window):
    import torch
    q, k, v = to_dev(x["q"]), to_dev(x["k"]), to_dev(x["v"])
    cu = cu_dev(x["cu"])
    o, lse = fa.attention_forward(q, k, v, causal=causal, window=window, scale=scale_of(d),
                                  cu_seqlens=cu, max_seqlen=N)
    fa.fa_device_status(torch.cuda.current_stream())
    return o, lse


@pytest.mark.parametrize("case", SMALL, ids=lambda c: f"B{c[0]}h{c[1]}x{c[2]}n{c[3]}d{c[4]}c{int(c[5])}w{c[6]}{'p' if c[7] else ''}")
def test_forward_matches_oracle(fa, oracle_mod, case):
    B, Hq, Hkv, N, d, causal, window, lengths = case
    x = make_case(B, Hq, Hkv, N, d, seed=7, lengths=lengths, with_dout=False)
    o, lse = run_fwd(fa, x, B, Hq, Hkv, N, d, causal, window)
    o_ref, lse_ref = oracle_mod.attention_fwd(x["q"], x["k"], x["v"], causal=causal,
                                              window=window, scale=scale_of(d),
                                              cu_seqlens=x["cu"])
    assert max_abs(to_f64(o), o_ref) <= O_MAX_ABS
    assert max_abs(lse.cpu().numpy().astype(np.float64), lse_ref) <= LSE_MAX_ABS


def test_forward_is_deterministic(fa):
    import torch
    x = make_case(2, 4, 2, 700, 128, seed=3, with_dout=False)
    o1, l1 = run_fwd(fa, x, 2, 4, 2, 700, 128, True, 0)
    o2, l2 = run_fwd(fa, x, 2, 4, 2, 700, 128, True, 0)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)


def test_forward_large_scores(fa, oracle_mod):
    """Scores spread over +-30 (q doubled, scale 0.5) move the running max by
    many units of log2, exercising the output rescale."""
    from exact_io_aware_tcgen05_gb300.inputs import bf16_bits_rne
    x = make_case(1, 2, 2, 640, 64, seed=11, with_dout=False)
    x["q"] = bf16_bits_rne(oracle_mod.to_f64(x["q"]).astype(np.float32) * 2)
    import torch
    q, k, v = to_dev(x["q"]), to_dev(x["k"]), to_dev(x["v"])
    o, lse = fa.attention_forward(q, k, v, causal=True, scale=0.5)
    fa.fa_device_status(torch.cuda.current_stream())
    o_ref, lse_ref = oracle_mod.attention_fwd(x["q"], x["k"], x["v"], causal=True, window=0,
                                              scale=0.5)
    assert np.isfinite(to_f64(o)).all()
    assert max_abs(to_f64(o), o_ref) <= O_MAX_ABS
    assert max_abs(lse.cpu().numpy().astype(np.float64), lse_ref) <= LSE_MAX_ABS


# A forward CTA may serve several consecutive query heads (fa_fwd_set_heads; those of
# one key/value group share its K/V tiles).  Every divisor of Hq, including counts that
# span several groups, must give the same bits, and they must match the oracle.
# (B, Hq, Hkv, N, d, causal, window, lengths, dtype)
HEADS_CASES = [
    (2, 8, 2, 300, 128, True, 0, None, "bf16"),
    (1, 8, 1, 700, 64, True, 200, None, "bf16"),                    # MQA, window
    (5, 4, 1, 513, 128, False, 0, (1, 127, 0, 129, 513), "f16"),     # packed, empty seq
    (3, 6, 2, 260, 64, True, 0, (260, 1, 131), "bf16"),              # group of 3
    (1, 4, 1, 100, 128, True, 0, None, "bf16"),                      # one key block per CTA
    (2, 8, 8, 300, 128, True, 0, None, "bf16"),                      # MHA
    (4, 4, 4, 300, 64, False, 0, (300, 1, 0, 129), "f16"),           # MHA, packed
]


@pytest.mark.parametrize("case", HEADS_CASES,
                         ids=lambda c: f"B{c[0]}h{c[1]}x{c[2]}n{c[3]}d{c[4]}c{int(c[5])}w{c[6]}"
                                       f"{'p' if c[7] else ''}{c[8]}")
def test_heads_per_cta_give_the_same_bits(fa, oracle_mod, case):
    import torch
    B, Hq, Hkv, N, d, causal, window, lengths, dtype = case
    x = make_case(B, Hq, Hkv, N, d, seed=62, lengths=lengths, dtype=dtype, with_dout=False)
    q, k, v = (to_dev(x[n]) for n in ("q", "k", "v"))
    kw = dict(causal=causal, window=window, scale=scale_of(d), cu_seqlens=cu_dev(x["cu"]),
              max_seqlen=N)
    first = None
    for heads in [c for c in range(1, Hq + 1) if Hq % c == 0]:
        o, lse = fa.attention_forward(q, k, v, heads=heads, **kw)
        fa.fa_device_status(torch.cuda.current_stream())
        if first is None:
            first = (o, lse)
            continue
        assert torch.equal(o.view(torch.int16), first[0].view(torch.int16)), heads
        assert torch.equal(lse, first[1]), heads
    o_ref, lse_ref = oracle_mod.attention_fwd(x["q"], x["k"], x["v"], causal=causal, window=window,
                                              scale=scale_of(d), cu_seqlens=x["cu"])
    assert max_abs(to_f64(first[0]), o_ref) <= O_MAX_ABS
    assert max_abs(first[1].cpu().numpy().astype(np.float64), lse_ref) <= LSE_MAX_ABS
