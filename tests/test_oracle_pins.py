"""Pins for the fp64 oracle, none of which uses the oracle to check itself.

Each test fixes the oracle's output by something other than its own formula:
hand-derived values, closed forms, invariants of softmax attention, fp64
finite differences, reductions between cases, and independent library
routines (PyTorch CPU fp64 scaled_dot_product_attention / autograd).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")


def rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def visible_mask(L, causal, window):
    i = np.arange(L)[:, None]
    j = np.arange(L)[None, :]
    m = np.ones((L, L), bool)
    if causal:
        m &= j <= i
    if window > 0:
        m &= (i - j) < window
    return m


MASKS = [(False, 0), (True, 0), (True, 1), (True, 3), (True, 7)]


# ------------------------------------------------------------ hand-derived

def test_hand_cases_forward(oracle_mod):
    g = json.load(open(GOLDEN))
    q = np.array(g["q"])[None]
    k, v = np.array(g["k"]), np.array(g["v"])
    for case in g["cases"]:
        o, lse = oracle_mod.fwd_group(q, k, v, case["causal"], case["window"], 1.0)
        np.testing.assert_allclose(o[0], case["o"], rtol=0, atol=1e-14, err_msg=case["name"])
        np.testing.assert_allclose(lse[0], case["lse"], rtol=0, atol=1e-14, err_msg=case["name"])


def test_hand_case_backward(oracle_mod):
    g = json.load(open(GOLDEN))
    q = np.array(g["q"])[None]
    k, v = np.array(g["k"]), np.array(g["v"])
    gc = g["grad_case"]
    dq, dk, dv = oracle_mod.bwd_group(q, k, v, np.array(gc["dout"])[None], gc["causal"],
                                      gc["window"], 1.0)
    np.testing.assert_allclose(dq[0], gc["dq"], atol=1e-14)
    np.testing.assert_allclose(dk, gc["dk"], atol=1e-14)
    np.testing.assert_allclose(dv, gc["dv"], atol=1e-14)


# ------------------------------------------------------------ closed forms

@pytest.mark.parametrize("causal,window", MASKS)
def test_constant_value_rows_give_that_constant(oracle_mod, causal, window):
    """All rows of V equal c  =>  O_i = c (the probabilities of a row sum to 1)."""
    G, L, d = 3, 37, 5
    c = rand(d, 1)
    q, k = rand((G, L, d), 2), rand((L, d), 3)
    v = np.tile(c, (L, 1))
    o, _ = oracle_mod.fwd_group(q, k, v, causal, window, 0.7)
    np.testing.assert_allclose(o, np.broadcast_to(c, o.shape), rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal,window", MASKS)
def test_zero_queries_give_mean_of_visible_values(oracle_mod, causal, window):
    """Q = 0 => S = 0 => uniform softmax: O_i = mean of v_j over the visible keys,
    LSE_i = ln |visible(i)| (global mean, prefix means, windowed means)."""
    G, L, d = 2, 41, 6
    q = np.zeros((G, L, d))
    k, v = rand((L, d), 4), rand((L, d), 5)
    o, lse = oracle_mod.fwd_group(q, k, v, causal, window, 0.3)
    exp_o = np.empty((L, d))
    exp_lse = np.empty(L)
    for i in range(L):
        lo = max(0, i - window + 1) if window > 0 else 0
        hi = i if causal else L - 1
        exp_o[i] = v[lo:hi + 1].mean(axis=0)
        exp_lse[i] = math.log(hi - lo + 1)
    for g in range(G):
        np.testing.assert_allclose(o[g], exp_o, rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[g], exp_lse, rtol=0, atol=1e-13)


def test_single_key_sequence(oracle_mod):
    """L = 1: O_0 = v_0 and LSE_0 = S_00 = scale * q.k."""
    q, k, v = rand((2, 1, 8), 6), rand((1, 8), 7), rand((1, 8), 8)
    o, lse = oracle_mod.fwd_group(q, k, v, True, 0, 0.25)
    np.testing.assert_allclose(o[:, 0], np.broadcast_to(v[0], (2, 8)), atol=1e-15)
    np.testing.assert_allclose(lse[:, 0], 0.25 * (q[:, 0] @ k[0]), atol=1e-14)


@pytest.mark.parametrize("causal,window", MASKS)
def test_constant_value_rows_give_zero_q_and_k_gradients(oracle_mod, causal, window):
    """V rows equal c => dP_ij = dO_i.c = D_i => dS = 0 => dQ = 0 and dK = 0."""
    G, L, d = 2, 19, 4
    q, k, do = rand((G, L, d), 9), rand((L, d), 10), rand((G, L, d), 11)
    v = np.tile(rand(d, 12), (L, 1))
    dq, dk, _ = oracle_mod.bwd_group(q, k, v, do, causal, window, 0.5)
    assert np.abs(dq).max() < 1e-13
    assert np.abs(dk).max() < 1e-13


# ------------------------------------------------- independent library route

@pytest.mark.parametrize("causal,window", MASKS)
@pytest.mark.parametrize("L,d", [(1, 4), (13, 8), (64, 16), (130, 32)])
def test_matches_torch_sdpa_fp64(oracle_mod, causal, window, L, d):
    """PyTorch CPU fp64 scaled_dot_product_attention with an explicit boolean mask."""
    G, scale = 2, 1.0 / math.sqrt(d)
    q, k, v = rand((G, L, d), 13), rand((L, d), 14), rand((L, d), 15)
    o, lse = oracle_mod.fwd_group(q, k, v, causal, window, scale)
    tq = torch.from_numpy(q)[None]
    tk = torch.from_numpy(k)[None, None].expand(1, G, L, d)
    tv = torch.from_numpy(v)[None, None].expand(1, G, L, d)
    mask = torch.from_numpy(visible_mask(L, causal, window))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask,
                                                           scale=scale)
    np.testing.assert_allclose(o, ref[0].numpy(), rtol=0, atol=1e-12)
    s = (tq @ tk.transpose(-1, -2)) * scale
    ref_lse = torch.logsumexp(s.masked_fill(~mask, -math.inf), dim=-1)
    np.testing.assert_allclose(lse, ref_lse[0].numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal,window", MASKS)
def test_gradients_match_torch_autograd_fp64(oracle_mod, causal, window):
    G, L, d, scale = 2, 33, 8, 0.35
    q, k, v, do = rand((G, L, d), 16), rand((L, d), 17), rand((L, d), 18), rand((G, L, d), 19)
    dq, dk, dv = oracle_mod.bwd_group(q, k, v, do, causal, window, scale)
    tq = torch.tensor(q, requires_grad=True)
    tk = torch.tensor(k, requires_grad=True)
    tv = torch.tensor(v, requires_grad=True)
    mask = torch.from_numpy(visible_mask(L, causal, window))
    out = torch.nn.functional.scaled_dot_product_attention(
        tq[None], tk[None, None].expand(1, G, L, d), tv[None, None].expand(1, G, L, d),
        attn_mask=mask, scale=scale)
    (out[0] * torch.from_numpy(do)).sum().backward()
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=0, atol=1e-12)


# ------------------------------------------------------------- invariants

@pytest.mark.parametrize("causal,window", MASKS)
def test_probabilities_from_lse_reproduce_output(oracle_mod, causal, window):
    """P_ij = exp(S_ij - LSE_i) is a probability row (sums to 1, zero outside the mask)
    and P V reproduces O: the identity the backward pass relies on."""
    G, L, d, scale = 2, 50, 8, 0.4
    q, k, v = rand((G, L, d), 20), rand((L, d), 21), rand((L, d), 22)
    o, lse = oracle_mod.fwd_group(q, k, v, causal, window, scale)
    mask = visible_mask(L, causal, window)
    for g in range(G):
        s = scale * q[g] @ k.T
        p = np.where(mask, np.exp(s - lse[g][:, None]), 0.0)
        np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-13)
        assert (p >= 0).all()
        np.testing.assert_allclose(p @ v, o[g], rtol=0, atol=1e-13)


def test_lse_independent_of_summation_order(oracle_mod):
    """LSE_i = ln sum_j exp(S_ij), recomputed with ascending-sorted summation."""
    G, L, d, scale = 1, 200, 16, 0.25
    q, k, v = rand((G, L, d), 23), rand((L, d), 24), rand((L, d), 25)
    _, lse = oracle_mod.fwd_group(q, k, v, True, 0, scale)
    for i in range(L):
        s = np.sort(scale * k[:i + 1] @ q[0, i])
        m = s.max()
        assert abs(lse[0, i] - (m + math.log(math.fsum(np.exp(s - m))))) < 1e-12


@pytest.mark.parametrize("causal,window", MASKS)
def test_gradient_sum_invariants(oracle_mod, causal, window):
    """sum_j dK_j = 0 (shifting every key by a constant vector shifts a row's scores
    equally); sum_j dV_j = sum over heads and rows of dO_i (probability rows sum to 1)."""
    G, L, d = 3, 29, 6
    q, k, v, do = rand((G, L, d), 26), rand((L, d), 27), rand((L, d), 28), rand((G, L, d), 29)
    dq, dk, dv = oracle_mod.bwd_group(q, k, v, do, causal, window, 0.6)
    np.testing.assert_allclose(dk.sum(axis=0), 0.0, atol=1e-12)
    np.testing.assert_allclose(dv.sum(axis=0), do.sum(axis=(0, 1)), atol=1e-12)


# -------------------------------------------------------- finite differences

@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 4)])
def test_gradients_match_finite_differences(oracle_mod, causal, window):
    """Central differences (h = 1e-6) of the loss <dO, O(Q, K, V)> in fp64."""
    G, L, d, scale, h = 2, 9, 4, 0.8, 1e-6
    q, k, v, do = rand((G, L, d), 30), rand((L, d), 31), rand((L, d), 32), rand((G, L, d), 33)
    dq, dk, dv = oracle_mod.bwd_group(q, k, v, do, causal, window, scale)

    def loss(qq, kk, vv):
        o, _ = oracle_mod.fwd_group(qq, kk, vv, causal, window, scale)
        return float((o * do).sum())

    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        fd = np.empty_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = xp, xm
            fd[idx] = (loss(args_p["q"], args_p["k"], args_p["v"])
                       - loss(args_m["q"], args_m["k"], args_m["v"])) / (2 * h)
        rel = np.linalg.norm(fd - g) / np.linalg.norm(g)
        assert rel < 1e-7, (name, rel)


# -------------------------------------------------- the online recurrence

@pytest.mark.parametrize("causal,window", MASKS + [(True, 64)])
@pytest.mark.parametrize("Br,Bc", [(1, 1), (4, 7), (16, 16), (128, 128), (33, 64)])
def test_block_recurrence_equals_definition(oracle_mod, causal, window, Br, Bc):
    """The online-softmax block recurrence (any block sizes, ragged tails) gives the
    same O and LSE as the plain definition."""
    G, L, d, scale = 2, 131, 8, 0.5
    q, k, v = rand((G, L, d), 34), rand((L, d), 35), rand((L, d), 36)
    o, lse = oracle_mod.fwd_group(q, k, v, causal, window, scale)
    ot, lset = oracle_mod.fwd_tiled_group(q, k, v, causal, window, scale, Br, Bc)
    np.testing.assert_allclose(ot, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lset, lse, rtol=0, atol=1e-12)


def test_block_recurrence_handles_large_scores(oracle_mod):
    """Scores near 700 would overflow exp without the max subtraction."""
    G, L, d = 1, 40, 2
    q = np.full((G, L, d), 20.0)
    k = np.abs(rand((L, d), 37)) * 20
    v = rand((L, d), 38)
    o, lse = oracle_mod.fwd_group(q, k, v, True, 0, 1.0)
    ot, lset = oracle_mod.fwd_tiled_group(q, k, v, True, 0, 1.0, 8, 8)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    np.testing.assert_allclose(ot, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lset, lse, rtol=1e-15, atol=1e-10)


# ------------------------------------------------------- reductions

def test_gqa_equals_repeated_heads(oracle_mod):
    """GQA equals multi-head attention with K, V repeated over each group; dK, dV are
    the group sums of the repeated heads' gradients."""
    B, N, Hq, Hkv, d = 2, 23, 8, 2, 8
    rng = np.random.default_rng(40)
    q, do = rng.standard_normal((B, N, Hq, d)), rng.standard_normal((B, N, Hq, d))
    k, v = rng.standard_normal((B, N, Hkv, d)), rng.standard_normal((B, N, Hkv, d))
    kw = dict(causal=True, window=5, scale=0.3)
    o, lse = oracle_mod.attention_fwd(q, k, v, **kw)
    kr, vr = np.repeat(k, Hq // Hkv, axis=2), np.repeat(v, Hq // Hkv, axis=2)
    o2, lse2 = oracle_mod.attention_fwd(q, kr, vr, **kw)
    np.testing.assert_allclose(o, o2, atol=1e-14)
    np.testing.assert_allclose(lse, lse2, atol=1e-14)
    dq, dk, dv = oracle_mod.attention_bwd(q, k, v, do, **kw)
    dq2, dk2, dv2 = oracle_mod.attention_bwd(q, kr, vr, do, **kw)
    np.testing.assert_allclose(dq, dq2, atol=1e-13)
    np.testing.assert_allclose(dk, dk2.reshape(B, N, Hkv, Hq // Hkv, d).sum(3), atol=1e-13)
    np.testing.assert_allclose(dv, dv2.reshape(B, N, Hkv, Hq // Hkv, d).sum(3), atol=1e-13)


@pytest.mark.parametrize("lengths", [[5, 1, 17, 9], [5, 0, 1, 17, 0, 9, 0]])
def test_packed_batch_equals_independent_sequences(oracle_mod, lengths):
    """A packed batch equals one call per sequence (no attention across sequences);
    empty sequences add nothing and leave the others unchanged."""
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T, Hq, Hkv, d = int(cu[-1]), 4, 2, 8
    rng = np.random.default_rng(41)
    q, do = rng.standard_normal((T, Hq, d)), rng.standard_normal((T, Hq, d))
    k, v = rng.standard_normal((T, Hkv, d)), rng.standard_normal((T, Hkv, d))
    kw = dict(causal=True, window=0, scale=0.4)
    o, lse = oracle_mod.attention_fwd(q, k, v, cu_seqlens=cu, **kw)
    dq, dk, dv = oracle_mod.attention_bwd(q, k, v, do, cu_seqlens=cu, **kw)
    for b, L in enumerate(lengths):
        if L == 0:
            continue
        s = slice(cu[b], cu[b + 1])
        ob, lb = oracle_mod.attention_fwd(q[s][None], k[s][None], v[s][None], **kw)
        np.testing.assert_allclose(o[s], ob[0], atol=1e-14)
        np.testing.assert_allclose(lse[:, s], lb[0], atol=1e-14)
        gq, gk, gv = oracle_mod.attention_bwd(q[s][None], k[s][None], v[s][None], do[s][None],
                                              **kw)
        np.testing.assert_allclose(dq[s], gq[0], atol=1e-14)
        np.testing.assert_allclose(dk[s], gk[0], atol=1e-14)
        np.testing.assert_allclose(dv[s], gv[0], atol=1e-14)


def test_window_at_least_length_equals_causal(oracle_mod):
    G, L, d = 2, 30, 8
    q, k, v, do = rand((G, L, d), 42), rand((L, d), 43), rand((L, d), 44), rand((G, L, d), 45)
    a = oracle_mod.fwd_group(q, k, v, True, L, 0.5)
    b = oracle_mod.fwd_group(q, k, v, True, 0, 0.5)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])
    ga = oracle_mod.bwd_group(q, k, v, do, True, L + 5, 0.5)
    gb = oracle_mod.bwd_group(q, k, v, do, True, 0, 0.5)
    for x, y in zip(ga, gb):
        np.testing.assert_array_equal(x, y)


def test_row_and_key_subsets_match_full(oracle_mod):
    """The sampled-row entry points return exactly the corresponding full-call rows."""
    G, L, d = 2, 45, 8
    q, k, v, do = rand((G, L, d), 46), rand((L, d), 47), rand((L, d), 48), rand((G, L, d), 49)
    rows = [44, 0, 17, 17, 3]
    o, lse = oracle_mod.fwd_group(q, k, v, True, 9, 0.5)
    os_, lses = oracle_mod.fwd_group(q, k, v, True, 9, 0.5, rows=rows)
    np.testing.assert_array_equal(os_, o[:, rows])
    np.testing.assert_array_equal(lses, lse[:, rows])
    dq, dk, dv = oracle_mod.bwd_group(q, k, v, do, True, 9, 0.5)
    krows = [1, 44, 30]
    sq, sk, sv = oracle_mod.bwd_group(q, k, v, do, True, 9, 0.5, qrows=rows, krows=krows)
    np.testing.assert_array_equal(sq, dq[:, rows])
    np.testing.assert_array_equal(sk, dk[krows])
    np.testing.assert_array_equal(sv, dv[krows])


def test_bf16_decode_is_exact(oracle_mod):
    from exact_io_aware_tcgen05_gb300.inputs import bf16_bits_rne
    x = np.array([1.0, -2.5, 3.140625, 0.0, 1e-3], np.float32)
    bits = bf16_bits_rne(x)
    back = oracle_mod.to_f64(bits)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(back, ref)


def test_f16_decode_is_exact(oracle_mod):
    """IEEE binary16 bit patterns decode to the values the format defines (sign,
    5-bit exponent with bias 15, 10-bit fraction, subnormals at exponent 0),
    worked out by hand here, not by numpy's own float16 conversion."""
    cases = {
        0x3C00: 1.0,                     # 2^0
        0xC000: -2.0,                    # sign, 2^1
        0x7BFF: 65504.0,                 # largest finite: (2 - 2^-10) * 2^15
        0x0400: 2.0 ** -14,              # smallest normal
        0x0001: 2.0 ** -24,              # smallest subnormal: 2^-10 * 2^-14
        0x3555: (1 + 0x155 / 1024) * 2.0 ** -2,   # 0.333251953125
        0x8000: -0.0,
    }
    bits = np.array(list(cases), dtype=np.uint16)
    got = oracle_mod.to_f64(bits.view(np.float16))
    np.testing.assert_array_equal(got, np.array(list(cases.values())))
    assert np.signbit(got[-1])


def test_f16_inputs_round_to_nearest_even(oracle_mod):
    """The fp16 input draws are the float32 draws rounded to nearest, ties to even:
    check against the rounding written out on the bit patterns."""
    from exact_io_aware_tcgen05_gb300.inputs import normal_f16
    x32 = np.random.default_rng(4).standard_normal(size=4096, dtype=np.float32)
    got = oracle_mod.to_f64(normal_f16(4096, 4))
    # |x| < 65504 and, for these draws, >= 2^-14 or exactly representable: round the
    # 23-bit fraction to 10 bits by hand (normal range) and compare
    u = x32.view(np.uint32).astype(np.int64)
    sign = np.where(u >> 31, -1.0, 1.0)
    e = ((u >> 23) & 0xFF) - 127
    frac = (u & 0x7FFFFF) | 0x800000            # 24-bit significand
    normal = e >= -14
    shift = np.where(normal, 13, 13 + (-14 - e))  # bits dropped below fp16's last place
    shift = np.minimum(shift, 40)
    q = frac >> shift
    rem = frac - (q << shift)
    half = np.int64(1) << (shift - 1)
    q = q + ((rem > half) | ((rem == half) & ((q & 1) == 1)))
    ref = sign * q.astype(np.float64) * 2.0 ** (e - 23 + shift)
    np.testing.assert_array_equal(got, ref)
