"""The fp8 (e4m3) forward (fa_fp8_quantize_qk / fa_fp8_quantize_v / fa_fwd_fp8)
against the fp8 oracle.

Both sides start from the same seeded bf16 inputs and quantise them on their own;
the codes and scales must agree bit for bit (float32 division and e4m3 rounding
to nearest even on both sides).  The forward is then compared with exact
attention on the dequantised values: LSE within the bf16 path's 1e-3, O within
the per-element bound of oracle.fp8.o_error_bound (the kernel rounds P to e4m3
for the P V product).
"""
import numpy as np
import pytest

from helpers import LSE_MAX_ABS, cu_dev, make_case, scale_of, to_dev, to_f64

pytestmark = pytest.mark.gpu

# (B, Hq, Hkv, N, causal, window, lengths); d = 128
CASES = [
    (1, 1, 1, 128, False, 0, None),
    (2, 4, 2, 300, True, 0, None),
    (1, 8, 1, 700, True, 200, None),
    (6, 4, 2, 513, True, 0, (1, 127, 128, 129, 300, 513)),
    (3, 2, 1, 900, False, 0, (900, 5, 256)),
    (4, 2, 1, 300, True, 0, (300, 0, 17, 0)),     # empty sequences
]
D = 128


def _ids(c):
    return f"B{c[0]}h{c[1]}x{c[2]}n{c[3]}c{int(c[4])}w{c[5]}{'p' if c[6] else ''}"


def _gpu(fa, x, N, causal, window):
    import torch
    q, k, v = to_dev(x["q"]), to_dev(x["k"]), to_dev(x["v"])
    cu = cu_dev(x["cu"])
    ops = fa.quantize_fp8(q, k, v, cu_seqlens=cu, max_seqlen=N)
    o, lse = fa.attention_forward_fp8(ops, causal=causal, window=window, scale=scale_of(D),
                                      cu_seqlens=cu, max_seqlen=N)
    fa.fa_device_status(torch.cuda.current_stream())
    assert o.dtype == torch.bfloat16
    return ops, o, lse


def _oracle_ops(fp8, x, B, N, nb, vt_tokens):
    cu = None if x["cu"] is None else [int(c) for c in x["cu"]]
    q8, qs = fp8.quantize_qk(x["q"], B, N, cu, nb=nb)
    k8, ks = fp8.quantize_qk(x["k"], B, N, cu, nb=nb)
    vt8, vs = fp8.quantize_v(x["v"], B, N, cu, vt_tokens=vt_tokens)
    return cu, (q8, qs, k8, ks, vt8, vs)


def _check_quantisation(fp8, ops, ref, B, N, cu):
    q8, qs, k8, ks, vt8, vs = (t.cpu().numpy() for t in ops[:6])
    rq8, rqs, rk8, rks, rvt8, rvs = ref
    # the columns the layout assigns to the sequences' blocks (a packed batch leaves
    # unused columns between sequences)
    offs, _ = fp8.block_offsets(B, N, cu)
    used = np.concatenate([np.arange(o, o + -(-L // 128)) for o, (_, L) in
                           zip(offs, fp8.seq_lengths(B, N, cu))]).astype(np.int64)
    assert np.array_equal(q8, rq8) and np.array_equal(k8, rk8)
    assert np.array_equal(qs[:, used], rqs[:, used])
    assert np.array_equal(ks[:, used], rks[:, used])
    assert np.array_equal(vs, rvs)
    cols = (128 * used[:, None] + np.arange(128)[None, :]).ravel()   # padding included
    assert np.array_equal(vt8[:, :, cols], rvt8[:, :, cols])


def _check_forward(fp8, x, ref, o, lse, B, Hq, Hkv, N, causal, window, cu, rows_per_seq=None,
                   fro_max=4e-2):
    q8, qs, k8, ks, vt8, vs = ref
    qd = fp8.dequantize_qk(q8, qs, B, N, cu)
    kd = fp8.dequantize_qk(k8, ks, B, N, cu)
    vd = fp8.dequantize_v(vt8, vs, B, N, cu)
    og, lg = to_f64(o), lse.cpu().numpy().astype(np.float64)
    G = Hq // Hkv
    import oracle
    worst, err2, ref2 = -np.inf, 0.0, 0.0
    for b, (start, L) in enumerate(fp8.seq_lengths(B, N, cu)):
        if L == 0:
            continue            # an empty sequence has no rows (its scales are checked above)
        rows = np.arange(L) if rows_per_seq is None else np.unique(np.clip(rows_per_seq, 0, L - 1))
        qs_, ks_, vs_ = ((qd[b], kd[b], vd[b]) if cu is None else
                         (qd[start:start + L], kd[start:start + L], vd[start:start + L]))
        for h in range(Hq):
            qh, kg, vg = qs_[:, h], ks_[:, h // G], vs_[:, h // G]
            o_ref, l_ref = oracle.fwd_group(qh[None], kg, vg, causal, window, scale_of(D), rows=rows)
            o_ref, l_ref = o_ref[0], l_ref[0]
            if cu is None:
                o_got, l_got = og[b, rows, h], lg[b, h, rows]
            else:
                o_got, l_got = og[start + rows, h], lg[h, start + rows]
            assert np.max(np.abs(l_got - l_ref)) <= LSE_MAX_ABS
            lse_full = np.zeros(L)
            lse_full[rows] = l_ref
            bound = fp8.o_error_bound(qh, kg, vg, lse_full, causal=causal, window=window,
                                      scale=scale_of(D), rows=rows)
            worst = max(worst, float(np.max(np.abs(o_got - o_ref) - bound)))
            err2 += float(np.sum((o_got - o_ref) ** 2))
            ref2 += float(np.sum(o_ref ** 2))
    assert worst <= 0.0, f"O outside the e4m3 bound by {worst}"
    if fro_max is None:
        return
    # statistical check on N(0,1) inputs.  Rounding a value spread over a binade to e4m3
    # (spacing 2^-3 of the binade's base) leaves an RMS relative error of about
    # 2^-3 ln 2 / sqrt(12) ~ 2.5%; with diffuse attention O and its error both shrink
    # like 1 / sqrt(keys seen), so the relative Frobenius error of O sits near that
    # figure.  4% leaves room for the sampling spread and catches a doubled error.
    assert np.sqrt(err2 / ref2) <= fro_max


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_fp8_quantisation_and_forward_match_oracle(fa, oracle_mod, case):
    from oracle import fp8
    B, Hq, Hkv, N, causal, window, lengths = case
    x = make_case(B, Hq, Hkv, N, D, seed=31, lengths=lengths, with_dout=False)
    ops, o, lse = _gpu(fa, x, N, causal, window)
    cu, ref = _oracle_ops(fp8, x, B if lengths is None else len(lengths), N, ops.nb, ops.vt_tokens)
    Bn = B if lengths is None else len(lengths)
    _check_quantisation(fp8, ops, ref, Bn, N, cu)
    _check_forward(fp8, x, ref, o, lse, Bn, Hq, Hkv, N, causal, window, cu)


def test_fp8_fullsize_sampled_rows(fa, oracle_mod):
    """B2 H16 N8192 d128 causal (the bench shape): quantisation checked everywhere,
    the forward on sampled rows of every head."""
    from oracle import fp8
    B, Hq, Hkv, N = 2, 16, 16, 8192
    x = make_case(B, Hq, Hkv, N, D, seed=0, with_dout=False)
    ops, o, lse = _gpu(fa, x, N, True, 0)
    cu, ref = _oracle_ops(fp8, x, B, N, ops.nb, ops.vt_tokens)
    _check_quantisation(fp8, ops, ref, B, N, cu)
    rows = np.array([0, 1, 127, 128, 255, 256, 4095, 4096, 8190, 8191])
    _check_forward(fp8, x, ref, o, lse, B, Hq, Hkv, N, True, 0, cu, rows_per_seq=rows)


def test_fp8_rejects_d64_and_short_buffers(fa):
    import torch
    dev = "cuda"
    q8 = torch.zeros((1, 128, 1, 64), dtype=torch.uint8, device=dev)
    sc = torch.ones((1, 1), dtype=torch.float32, device=dev)
    vt = torch.zeros((1, 64, 128), dtype=torch.uint8, device=dev)
    o = torch.empty((1, 128, 1, 64), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((1, 1, 128), dtype=torch.float32, device=dev)
    st = fa.fa_fwd_fp8(q8, sc, q8, sc, vt, sc, 1, 128, o, lse, 1, 1, 1, 128, 64, 0, 0, None, 0,
                       0.125, check=False)
    assert st == fa.FA_ERR_UNSUPPORTED
    q8 = torch.zeros((1, 300, 1, 128), dtype=torch.uint8, device=dev)
    o = torch.empty((1, 300, 1, 128), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((1, 1, 300), dtype=torch.float32, device=dev)
    vt = torch.zeros((1, 128, 384), dtype=torch.uint8, device=dev)
    sc3 = torch.ones((1, 3), dtype=torch.float32, device=dev)
    # nb = 2 < 3 blocks; vt_tokens = 256 < 384
    assert fa.fa_fwd_fp8(q8, sc3, q8, sc3, vt, sc, 2, 384, o, lse, 1, 1, 1, 300, 128, 0, 0, None, 0,
                         0.1, check=False) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_fp8(q8, sc3, q8, sc3, vt, sc, 3, 256, o, lse, 1, 1, 1, 300, 128, 0, 0, None, 0,
                         0.1, check=False) == fa.FA_ERR_INVALID_ARG


# ------------------------------------------------------ incoherent processing
#
# fa_fp8_quantize_qk_incoherent rotates every row of Q and K by
# (1/sqrt d) H diag(sigma) before the block quantisation.  The codes and scales must
# equal the oracle's bit for bit (the same float32 operations in the same order), V
# is untouched, and the unchanged fp8 forward on the rotated operands is exact
# attention on their dequantised values within the same e4m3 bound as above.

def _with_outliers(x, amp=16.0, channels=(3, 77)):
    """The inputs incoherent processing is for: Q and K with a few channels amp times
    the others (a power of two, so the bf16 values stay exact)."""
    out = dict(x)
    for name in ("q", "k"):
        f = (x[name].astype(np.uint32) << 16).view(np.float32).copy()
        f[..., [c % f.shape[-1] for c in channels]] *= np.float32(amp)
        out[name] = (f.view(np.uint32) >> 16).astype(np.uint16)
    return out


# (B, Hq, Hkv, N, causal, window, lengths, seed); d = 128
ROT_CASES = [
    (1, 1, 1, 128, False, 0, None, 5),
    (2, 4, 2, 300, True, 0, None, (3 << 32) | 17),          # both key words of the seed
    (6, 4, 2, 513, True, 0, (1, 127, 128, 129, 300, 513), 99),
    (4, 2, 1, 300, True, 0, (300, 0, 17, 0), 12345),          # empty sequences
]


def _rot_ops(fa, fp8, x, N, nb_B, seed):
    cu = cu_dev(x["cu"])
    q, k, v = to_dev(x["q"]), to_dev(x["k"]), to_dev(x["v"])
    ops = fa.quantize_fp8(q, k, v, cu_seqlens=cu, max_seqlen=N, incoherent_seed=seed)
    cu_l = None if x["cu"] is None else [int(c) for c in x["cu"]]
    ref = (*fp8.quantize_qk(x["q"], nb_B, N, cu_l, nb=ops.nb, rotate_seed=seed),
           *fp8.quantize_qk(x["k"], nb_B, N, cu_l, nb=ops.nb, rotate_seed=seed),
           *fp8.quantize_v(x["v"], nb_B, N, cu_l, vt_tokens=ops.vt_tokens))
    return ops, ref, cu, cu_l


@pytest.mark.parametrize("case", ROT_CASES, ids=lambda c: _ids(c[:7]) + f"s{c[7]}")
def test_fp8_incoherent_quantisation_and_forward_match_oracle(fa, oracle_mod, case):
    from oracle import fp8
    import torch
    B, Hq, Hkv, N, causal, window, lengths, seed = case
    x = _with_outliers(make_case(B, Hq, Hkv, N, D, seed=41, lengths=lengths, with_dout=False))
    Bn = B if lengths is None else len(lengths)
    ops, ref, cu, cu_l = _rot_ops(fa, fp8, x, N, Bn, seed)
    o, lse = fa.attention_forward_fp8(ops, causal=causal, window=window, scale=scale_of(D),
                                      cu_seqlens=cu, max_seqlen=N)
    fa.fa_device_status(torch.cuda.current_stream())
    _check_quantisation(fp8, ops, ref, Bn, N, cu_l)
    _check_forward(fp8, x, ref, o, lse, Bn, Hq, Hkv, N, causal, window, cu_l)


@pytest.mark.parametrize("lengths", [None, (1, 200, 64, 0, 129)], ids=["dense", "packed"])
def test_fp8_incoherent_quantisation_d64(fa, oracle_mod, lengths):
    # the quantisers also take d = 64 (three butterfly stages between lanes, not two)
    from oracle import fp8
    B, H, N = 3, 2, 300
    x = _with_outliers(make_case(B, H, H, N, 64, seed=43, lengths=lengths, with_dout=False))
    Bn = B if lengths is None else len(lengths)
    ops, ref, _, cu_l = _rot_ops(fa, fp8, x, N if lengths is None else max(lengths), Bn, 0xABCDEF)
    _check_quantisation(fp8, ops, ref, Bn, N if lengths is None else max(lengths), cu_l)


def test_fp8_incoherent_fullsize_sampled_rows(fa, oracle_mod):
    """B2 H16 N8192 d128 causal with outlier channels: rotated codes and scales checked
    everywhere, the forward on sampled rows of every head."""
    from oracle import fp8
    B, Hq, Hkv, N = 2, 16, 16, 8192
    x = _with_outliers(make_case(B, Hq, Hkv, N, D, seed=0, with_dout=False))
    ops, ref, cu, cu_l = _rot_ops(fa, fp8, x, N, B, 2027)
    o, lse = fa.attention_forward_fp8(ops, causal=True, scale=scale_of(D))
    _check_quantisation(fp8, ops, ref, B, N, cu_l)
    rows = np.array([0, 1, 127, 128, 255, 256, 4095, 4096, 8190, 8191])
    _check_forward(fp8, x, ref, o, lse, B, Hq, Hkv, N, True, 0, cu_l, rows_per_seq=rows)


# ------------------------------------------------------------ random sweep
#
# Seeded random shapes through the fp8 path (d = 128): GQA group 1, 2 or 4; a dense
# batch or a packed one mixing empty, one- and two-token and longer sequences; causal or
# not, sometimes with a window; plain block quantisation or incoherent processing with
# a random 63-bit seed; Q and K with two channels 1x, 4x or 16x the others.  Codes and
# scales bit for bit, O within the per-element e4m3 bound, LSE within 1e-3 (the
# Frobenius check above is calibrated for long N(0,1) rows and is left out here).

def draw_fp8_cases(n, seed=2027):
    rng = np.random.default_rng(seed)
    cases = []
    for _ in range(n):
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
        rot = int(rng.integers(0, 2 ** 63)) if rng.random() < 0.5 else None
        amp = float(rng.choice([1.0, 4.0, 16.0]))
        cases.append((b, hq, hkv, n_max, causal, window, lengths, rot, amp))
    return cases


FP8_CASES = draw_fp8_cases(24)


def _fp8_id(c):
    b, hq, hkv, n, causal, window, lengths, rot, amp = c
    return (f"B{b}h{hq}x{hkv}n{n}c{int(causal)}w{window}{'p' if lengths else ''}"
            f"{'r' if rot is not None else ''}a{int(amp)}")


@pytest.mark.parametrize("idx", range(len(FP8_CASES)), ids=[_fp8_id(c) for c in FP8_CASES])
def test_fp8_random_shapes_match_oracle(fa, oracle_mod, idx):
    from oracle import fp8
    import torch
    b, hq, hkv, n, causal, window, lengths, rot, amp = FP8_CASES[idx]
    x = make_case(b, hq, hkv, n, D, seed=3000 + idx, lengths=lengths, with_dout=False)
    if amp != 1.0:
        x = _with_outliers(x, amp=amp)
    Bn = b if lengths is None else len(lengths)
    cu = cu_dev(x["cu"])
    q, k, v = to_dev(x["q"]), to_dev(x["k"]), to_dev(x["v"])
    ops = fa.quantize_fp8(q, k, v, cu_seqlens=cu, max_seqlen=n, incoherent_seed=rot)
    o, lse = fa.attention_forward_fp8(ops, causal=causal, window=window, scale=scale_of(D),
                                      cu_seqlens=cu, max_seqlen=n)
    fa.fa_device_status(torch.cuda.current_stream())
    cu_l = None if x["cu"] is None else [int(c) for c in x["cu"]]
    ref = (*fp8.quantize_qk(x["q"], Bn, n, cu_l, nb=ops.nb, rotate_seed=rot),
           *fp8.quantize_qk(x["k"], Bn, n, cu_l, nb=ops.nb, rotate_seed=rot),
           *fp8.quantize_v(x["v"], Bn, n, cu_l, vt_tokens=ops.vt_tokens))
    _check_quantisation(fp8, ops, ref, Bn, n, cu_l)
    _check_forward(fp8, x, ref, o, lse, Bn, hq, hkv, n, causal, window, cu_l, fro_max=None)
