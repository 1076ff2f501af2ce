"""Dropout (fa_fwd_dropout / fa_bwd_dropout) on the GPU against the dropout oracle.

The keep masks are checked bit for bit through inputs that expose them: with
Q = 0 every visible key gets probability 1/|visible|, so O = Z V with V the
identity shows Z = P * keep * r column by column (forward kernel), and dV = Z^T dO
with dO the identity shows it for the dK/dV kernel.  The dQ kernel's mask is
checked through parity of dQ on random inputs.
"""
import numpy as np
import pytest

from helpers import (GRAD_REL_FRO, LSE_MAX_ABS, O_MAX_ABS, cu_dev, make_case, max_abs, rel_fro,
                     scale_of, to_dev, to_f64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def drop():
    from oracle import dropout
    return dropout


def _bf16(a):
    from exact_io_aware_tcgen05_gb300.inputs import bf16_bits_rne
    return bf16_bits_rne(np.asarray(a, dtype=np.float32))


def _fwd(fa, q, k, v, causal, window, dropout, cu=None, N=None):
    import torch
    o, lse = fa.attention_forward(to_dev(q), to_dev(k), to_dev(v), causal=causal, window=window,
                                  scale=scale_of(q.shape[-1]), cu_seqlens=cu_dev(cu), max_seqlen=N,
                                  dropout=dropout)
    fa.fa_device_status(torch.cuda.current_stream())
    return to_f64(o), lse.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 77)])
def test_forward_keep_mask_is_exact(fa, drop, causal, window):
    B, H, N, d = 2, 3, 256, 128
    p, seed, off = 0.3, 0xDEADBEEF12345678, 5
    rng = np.random.default_rng(0)
    q = _bf16(np.zeros((B, N, H, d)))
    k = _bf16(rng.standard_normal((B, N, H, d)))
    t = drop.threshold(p)
    r = 256.0 / (256 - t)
    for half in range(2):                     # keys 128 half .. + 127 on the 128 columns
        v = np.zeros((B, N, H, d), np.float32)
        for j in range(128):
            v[:, 128 * half + j, :, j] = 1.0
        o, _ = _fwd(fa, q, k, _bf16(v), causal, window, (p, seed, off))
        for b in range(B):
            for h in range(H):
                keep = drop.keep_mask(N, b * H + h, p, seed, off)
                vis = drop._visible(N, causal, window)
                nvis = vis.sum(axis=1, keepdims=True)
                keys = slice(128 * half, 128 * half + 128)
                z = o[b, :, h, :]                                   # [N, 128]
                expect = np.where(vis[:, keys] & keep[:, keys], r / nvis, 0.0)
                assert np.array_equal(z > 0.5 * r / nvis, expect > 0), (half, b, h)
                np.testing.assert_allclose(z, expect, rtol=1e-2, atol=1e-6)


def test_backward_dkdv_keep_mask_is_exact(fa, drop):
    """dV = Z^T dO with dO one-hot per query shows Z as the dK/dV kernel applies it."""
    import torch
    B, H, N, d = 1, 2, 256, 128
    p, seed, off = 0.5, 77, 9
    rng = np.random.default_rng(1)
    q = _bf16(np.zeros((B, N, H, d)))
    k = _bf16(rng.standard_normal((B, N, H, d)))
    v = _bf16(rng.standard_normal((B, N, H, d)))
    t = drop.threshold(p)
    r = 256.0 / (256 - t)
    vis = drop._visible(N, True, 0)
    nvis = vis.sum(axis=1, keepdims=True)
    for half in range(2):                     # queries 128 half .. + 127 on the columns
        dout = np.zeros((B, N, H, d), np.float32)
        for i in range(128):
            dout[:, 128 * half + i, :, i] = 1.0
        qd, kd, vd, dd = to_dev(q), to_dev(k), to_dev(v), to_dev(_bf16(dout))
        kw = dict(causal=True, dropout=(p, seed, off))
        o, lse = fa.attention_forward(qd, kd, vd, **kw)
        _, _, dv = fa.attention_backward(qd, kd, vd, o, lse, dd, **kw)
        fa.fa_device_status(torch.cuda.current_stream())
        dv = to_f64(dv)
        for h in range(H):
            keep = drop.keep_mask(N, h, p, seed, off)
            qs = slice(128 * half, 128 * half + 128)
            expect = np.where(vis[qs] & keep[qs], r / nvis[qs], 0.0).T     # [keys, 128 queries]
            got = dv[0, :, h, :]
            assert np.array_equal(got > 0.5 * (r / nvis[qs]).T, expect > 0), (half, h)
            np.testing.assert_allclose(got, expect, rtol=1e-2, atol=1e-6)


# (B, Hq, Hkv, N, d, causal, window, lengths)
CASES = [
    (2, 4, 2, 300, 128, True, 0, None),
    (1, 4, 4, 513, 64, True, 0, None),
    (1, 8, 1, 700, 128, True, 200, None),
    (2, 2, 2, 200, 128, False, 0, None),
    (2, 4, 2, 300, 64, False, 0, None),
    (6, 4, 2, 513, 128, True, 0, (1, 127, 128, 129, 300, 513)),
    (6, 4, 2, 513, 64, True, 0, (1, 127, 128, 129, 300, 513)),
]


@pytest.mark.parametrize("path", ["fused", "split"])
@pytest.mark.parametrize("p_drop", [0.1, 0.3])
@pytest.mark.parametrize("case", CASES, ids=lambda c: f"B{c[0]}h{c[1]}x{c[2]}n{c[3]}d{c[4]}c{int(c[5])}w{c[6]}{'p' if c[7] else ''}")
def test_dropout_matches_oracle(fa, drop, case, p_drop, path):
    import torch
    B, Hq, Hkv, N, d, causal, window, lengths = case
    x = make_case(B, Hq, Hkv, N, d, seed=31, lengths=lengths)
    seed, off = 123456789, 3
    kw = dict(causal=causal, window=window, scale=scale_of(d), cu_seqlens=cu_dev(x["cu"]),
              max_seqlen=N, dropout=(p_drop, seed, off))
    q, k, v, do = (to_dev(x[n]) for n in ("q", "k", "v", "dout"))
    o, lse = fa.attention_forward(q, k, v, **kw)
    dq, dk, dv = fa.attention_backward(q, k, v, o, lse, do, path=path, **kw)
    fa.fa_device_status(torch.cuda.current_stream())
    okw = dict(causal=causal, window=window, scale=scale_of(d), p_drop=p_drop, seed=seed,
               offset=off, cu_seqlens=x["cu"])
    o_ref, lse_ref = drop.attention_fwd(x["q"], x["k"], x["v"], **okw)
    assert max_abs(to_f64(o), o_ref) <= O_MAX_ABS
    assert max_abs(lse.cpu().numpy().astype(np.float64), lse_ref) <= LSE_MAX_ABS
    refs = drop.attention_bwd(x["q"], x["k"], x["v"], x["dout"], **okw)
    for name, g, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
        assert rel_fro(to_f64(g), ref) <= GRAD_REL_FRO, name


def test_zero_dropout_is_bitwise_the_plain_path(fa):
    import torch
    x = make_case(2, 4, 2, 300, 128, seed=8)
    q, k, v, do = (to_dev(x[n]) for n in ("q", "k", "v", "dout"))
    a = fa.attention_forward(q, k, v, causal=True)
    b = fa.attention_forward(q, k, v, causal=True, dropout=(0.0, 5, 1))
    ga = fa.attention_backward(q, k, v, a[0], a[1], do, causal=True)
    gb = fa.attention_backward(q, k, v, b[0], b[1], do, causal=True, dropout=(0.0, 5, 1))
    torch.cuda.synchronize()
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
    assert torch.equal(a[1], b[1])
    for u, w in zip(ga, gb):
        assert torch.equal(u.view(torch.int16), w.view(torch.int16))


def test_dropout_is_deterministic_and_offset_changes_the_mask(fa):
    import torch
    x = make_case(1, 4, 2, 400, 128, seed=9)
    q, k, v, do = (to_dev(x[n]) for n in ("q", "k", "v", "dout"))

    def run(off):
        kw = dict(causal=True, dropout=(0.2, 42, off))
        o, lse = fa.attention_forward(q, k, v, **kw)
        return (o,) + fa.attention_backward(q, k, v, o, lse, do, **kw)

    a, b, c = run(0), run(0), run(1)
    torch.cuda.synchronize()
    for u, w in zip(a, b):
        assert torch.equal(u.view(torch.int16), w.view(torch.int16))
    assert not torch.equal(a[0].view(torch.int16), c[0].view(torch.int16))
