"""fp64 CPU oracle for attention with dropout on the probabilities.

TEST INFRASTRUCTURE ONLY (same rules as the rest of ``oracle/``: only ``tests/``
and the measurement legs of ``bench.py`` may use it; it shares nothing with the
CUDA side).

The pages give dropout no semantics, so the definition is this library's own
(stated with the C ABI's dropout entry points):

* P is the masked softmax of S = scale * Q K^T (before dropout), LSE as without
  dropout.
* keep_ij in {0, 1} for query i, key j (positions within their sequence) of
  sequence b and query head h: the Philox4x32-10 call with counter
  (j // 4, i // 4, b * Hq + h, offset) and key (seed mod 2^32, seed // 2^32)
  returns four 32-bit words; byte j % 4 (bits 8 (j % 4) ..) of word i % 4 is
  the pair's byte, and keep_ij = (byte >= t), t = floor(256 p + 1/2) computed
  in float32.
* Z = P * keep * r with r = 256 / (256 - t);  O = Z V.
* Backward for the loss <dO, O> with keep fixed: dV = Z^T dO,
  dP = keep * r * (dO V^T), D_i = dO_i . O_i, dS = P * (dP - D),
  dQ = scale dS K, dK = scale dS^T Q (GQA: dK, dV summed over the group).

Philox4x32-10 follows its published definition: Salmon, Moraes, Dror, Shaw,
"Parallel Random Numbers: As Easy as 1, 2, 3" (SC 2011) -- ten rounds of
(c0, c1, c2, c3) -> (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1,
lo(M0 c0)), the key advanced by the Weyl increments between rounds.  Dense
matrices, one (sequence, head) at a time: for the small sizes tests use.
"""
from __future__ import annotations

import numpy as np

from . import _sequences, _take, _lse_shape, to_f64

_M0, _M1 = np.uint64(0xD2511F53), np.uint64(0xCD9E8D57)
_W0, _W1 = 0x9E3779B9, 0xBB67AE85
_MASK = np.uint64(0xFFFFFFFF)


def philox4x32_10(c0, c1, c2, c3, k0: int, k1: int):
    """Philox4x32-10 on arrays of uint32 counters (broadcast); returns 4 uint32 arrays."""
    c0, c1, c2, c3 = (np.asarray(c, dtype=np.uint64) & _MASK for c in (c0, c1, c2, c3))
    k0, k1 = int(k0) & 0xFFFFFFFF, int(k1) & 0xFFFFFFFF
    for r in range(10):
        if r > 0:
            k0 = (k0 + _W0) & 0xFFFFFFFF
            k1 = (k1 + _W1) & 0xFFFFFFFF
        p0 = _M0 * c0
        p1 = _M1 * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK
        c0, c1, c2, c3 = (hi1 ^ c1 ^ np.uint64(k0), lo1, hi0 ^ c3 ^ np.uint64(k1), lo0)
    return tuple(x.astype(np.uint32) for x in (c0, c1, c2, c3))


def threshold(p_drop: float) -> int:
    """t = floor(256 p + 1/2), evaluated in float32 like the library."""
    t = np.floor(np.float32(p_drop) * np.float32(256.0) + np.float32(0.5))
    return int(t)


def keep_mask(L: int, head_seq: int, p_drop: float, seed: int, offset: int) -> np.ndarray:
    """keep[i, j] (bool) for one (sequence, query head) of length L."""
    t = threshold(p_drop)
    nb = (L + 3) // 4
    I, J = np.meshgrid(np.arange(nb), np.arange(nb), indexing="ij")
    words = philox4x32_10(J, I, np.full_like(I, head_seq), np.full_like(I, offset),
                          seed & 0xFFFFFFFF, seed >> 32)
    w = np.stack(words, axis=-1)                         # [I, J, word = i % 4]
    i = np.arange(L)[:, None]
    j = np.arange(L)[None, :]
    word = w[i // 4, j // 4, i % 4].astype(np.uint64)
    byte = (word >> (8 * (j % 4)).astype(np.uint64)) & np.uint64(0xFF)
    return byte >= np.uint64(t)


def _visible(L: int, causal: bool, window: int) -> np.ndarray:
    i = np.arange(L)[:, None]
    j = np.arange(L)[None, :]
    vis = np.ones((L, L), dtype=bool)
    if causal:
        vis &= j <= i
        if window > 0:
            vis &= (i - j) < window
    return vis


def _softmax(s, vis):
    s = np.where(vis, s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    e = np.where(vis, np.exp(s - m_safe), 0.0)
    l = e.sum(axis=1, keepdims=True)
    p = np.divide(e, l, out=np.zeros_like(e), where=l > 0)
    lse = np.where(l[:, 0] > 0, m_safe[:, 0] + np.log(np.where(l[:, 0] > 0, l[:, 0], 1.0)), -np.inf)
    return p, lse


def attention_fwd(q, k, v, *, causal: bool, window: int, scale: float, p_drop: float, seed: int,
                  offset: int, cu_seqlens=None):
    """(O, LSE) in float64, layouts of the library."""
    q, k, v = to_f64(q), to_f64(k), to_f64(v)
    Hq, Hkv = q.shape[-2], k.shape[-2]
    G = Hq // Hkv
    t = threshold(p_drop)
    r = 256.0 / (256 - t)
    o = np.zeros(q.shape)
    lse = np.full(_lse_shape(q, Hq, cu_seqlens), -np.inf)
    for b, sel in _sequences(q, cu_seqlens):
        qs, ks, vs = _take(q, sel), _take(k, sel), _take(v, sel)
        L = qs.shape[0]
        vis = _visible(L, causal, window)
        for h in range(Hq):
            g = h // G
            p, l_h = _softmax(scale * qs[:, h] @ ks[:, g].T, vis)
            z = p * keep_mask(L, b * Hq + h, p_drop, seed, offset) * r
            oh = z @ vs[:, g]
            if sel[0] is not None:
                o[b, sel[1], h] = oh
                lse[b, h, sel[1]] = l_h
            else:
                o[sel[1], h] = oh
                lse[h, sel[1]] = l_h
    return o, lse


def attention_bwd(q, k, v, dout, *, causal: bool, window: int, scale: float, p_drop: float,
                  seed: int, offset: int, cu_seqlens=None):
    """(dQ, dK, dV) in float64 for the forward above."""
    q, k, v, dout = to_f64(q), to_f64(k), to_f64(v), to_f64(dout)
    Hq, Hkv = q.shape[-2], k.shape[-2]
    G = Hq // Hkv
    t = threshold(p_drop)
    r = 256.0 / (256 - t)
    dq, dk, dv = np.zeros(q.shape), np.zeros(k.shape), np.zeros(v.shape)
    for b, sel in _sequences(q, cu_seqlens):
        qs, ks, vs, ds = _take(q, sel), _take(k, sel), _take(v, sel), _take(dout, sel)
        L = qs.shape[0]
        vis = _visible(L, causal, window)
        for h in range(Hq):
            g = h // G
            p, _ = _softmax(scale * qs[:, h] @ ks[:, g].T, vis)
            kr = keep_mask(L, b * Hq + h, p_drop, seed, offset) * r
            z = p * kr
            o = z @ vs[:, g]
            dvh = z.T @ ds[:, h]
            dpm = kr * (ds[:, h] @ vs[:, g].T)
            dd = (ds[:, h] * o).sum(axis=1, keepdims=True)
            dsm = p * (dpm - dd)
            dqh = scale * dsm @ ks[:, g]
            dkh = scale * dsm.T @ qs[:, h]
            if sel[0] is not None:
                dq[b, sel[1], h] = dqh
                dk[b, sel[1], g] += dkh
                dv[b, sel[1], g] += dvh
            else:
                dq[sel[1], h] = dqh
                dk[sel[1], g] += dkh
                dv[sel[1], g] += dvh
    return dq, dk, dv
