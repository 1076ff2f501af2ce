"""Pins of the dropout oracle (oracle/dropout.py), against things other than itself."""
import numpy as np
import pytest

from helpers import make_case, scale_of


@pytest.fixture(scope="module")
def drop():
    from oracle import dropout
    return dropout


# Philox4x32-10 known-answer vectors published with the generator (Salmon et al.,
# "Parallel Random Numbers: As Easy as 1, 2, 3", Random123 test vectors):
# (counter, key) -> output
PHILOX_KAT = [
    ((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
    ((0xFFFFFFFF,) * 4, (0xFFFFFFFF, 0xFFFFFFFF), (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
     (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
]


@pytest.mark.parametrize("ctr,key,out", PHILOX_KAT)
def test_philox_known_answers(drop, ctr, key, out):
    got = drop.philox4x32_10(*[np.array([c]) for c in ctr], key[0], key[1])
    assert tuple(int(g[0]) for g in got) == out


def test_keep_mask_matches_elementwise_definition(drop):
    """The vectorised mask equals the definition applied pair by pair."""
    L, hs, p, seed, off = 11, 5, 0.3, 0x1234_5678_9ABC_DEF0, 7
    t = drop.threshold(p)
    keep = drop.keep_mask(L, hs, p, seed, off)
    for i in range(L):
        for j in range(L):
            words = drop.philox4x32_10(np.array([j // 4]), np.array([i // 4]), np.array([hs]),
                                       np.array([off]), seed & 0xFFFFFFFF, seed >> 32)
            byte = (int(words[i % 4][0]) >> (8 * (j % 4))) & 0xFF
            assert keep[i, j] == (byte >= t)


def test_threshold_rounds_to_nearest(drop):
    assert drop.threshold(0.0) == 0
    assert drop.threshold(0.1) == 26          # 25.6 -> 26
    assert drop.threshold(0.5) == 128
    assert drop.threshold(1.5 / 256) == 2     # ties round up (floor of x + 1/2)


def test_keep_fraction(drop):
    """Kept fraction of a large mask is (256 - t) / 256 within 6 standard deviations."""
    L = 2048
    for p in (0.1, 0.5):
        keep = drop.keep_mask(L, 3, p, 99, 0)
        q = (256 - drop.threshold(p)) / 256
        n = L * L
        assert abs(keep.mean() - q) < 6 * np.sqrt(q * (1 - q) / n)


@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 3)])
def test_zero_dropout_is_the_plain_oracle(drop, oracle_mod, causal, window):
    x = make_case(2, 4, 2, 37, 16, seed=3)
    kw = dict(causal=causal, window=window, scale=scale_of(16))
    o, lse = drop.attention_fwd(x["q"], x["k"], x["v"], p_drop=0.0, seed=1, offset=0, **kw)
    o_ref, lse_ref = oracle_mod.attention_fwd(x["q"], x["k"], x["v"], **kw)
    np.testing.assert_allclose(o, o_ref, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, atol=1e-12)
    g = drop.attention_bwd(x["q"], x["k"], x["v"], x["dout"], p_drop=0.0, seed=1, offset=0, **kw)
    g_ref = oracle_mod.attention_bwd(x["q"], x["k"], x["v"], x["dout"], **kw)
    for a, b in zip(g, g_ref):
        np.testing.assert_allclose(a, b, atol=1e-11)


def test_dropout_is_unbiased(drop, oracle_mod):
    """Averaged over seeds, the output approaches the output without dropout
    (the keep scaling r = 256 / (256 - t) is what makes it so)."""
    x = make_case(1, 1, 1, 24, 8, seed=5, with_dout=False)
    kw = dict(causal=True, window=0, scale=scale_of(8))
    o_ref, _ = oracle_mod.attention_fwd(x["q"], x["k"], x["v"], **kw)
    n = 400
    acc = np.zeros_like(o_ref)
    for s in range(n):
        o, _ = drop.attention_fwd(x["q"], x["k"], x["v"], p_drop=0.25, seed=s, offset=0, **kw)
        acc += o
    err = np.abs(acc / n - o_ref).max()
    assert err < 0.1 * np.abs(o_ref).max()
    # and a single draw is not the mean: dropout really drops
    o1, _ = drop.attention_fwd(x["q"], x["k"], x["v"], p_drop=0.25, seed=0, offset=0, **kw)
    assert np.abs(o1 - o_ref).max() > 0.05


def test_dropout_gradients_match_finite_differences(drop):
    """With the keep mask fixed by (seed, offset), O is differentiable; central
    differences of <dO, O> confirm dQ, dK, dV."""
    rng = np.random.default_rng(2)
    L, Hq, Hkv, d = 6, 2, 1, 3
    q = rng.standard_normal((1, L, Hq, d))
    k = rng.standard_normal((1, L, Hkv, d))
    v = rng.standard_normal((1, L, Hkv, d))
    do = rng.standard_normal((1, L, Hq, d))
    kw = dict(causal=True, window=0, scale=0.7, p_drop=0.3, seed=11, offset=2)

    def loss(q_, k_, v_):
        o, _ = drop.attention_fwd(q_, k_, v_, **kw)
        return float((o * do).sum())

    grads = drop.attention_bwd(q, k, v, do, **kw)
    eps = 1e-6
    for idx, (arr, g) in enumerate(zip((q, k, v), grads)):
        num = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            mi = it.multi_index
            a1, a2 = arr.copy(), arr.copy()
            a1[mi] += eps
            a2[mi] -= eps
            args1 = [q, k, v]
            args2 = [q, k, v]
            args1[idx], args2[idx] = a1, a2
            num[mi] = (loss(*args1) - loss(*args2)) / (2 * eps)
        np.testing.assert_allclose(g, num, atol=1e-6, rtol=1e-5)
