"""fp64 CPU oracle for the fp8 (e4m3) forward pass.

TEST INFRASTRUCTURE ONLY (same rules as the rest of ``oracle/``: only ``tests/``
and the measurement legs of ``bench.py`` may use it; it shares nothing with the
CUDA side).

The pages name FP8 only as a FlashAttention-3 capability ("block quantization"
of the inputs, "incoherent processing"; "FlashAttention: How IO-Aware Tiling
and Online Softmax Solved Transformer Memory Bottlenecks", "FlashAttention-3"
bullets) and give no format, block size or scale rule.  The definition below is
this library's own, stated with the C ABI's fp8 entry points.

* e4m3 is the 8-bit float with 1 sign bit, 4 exponent bits (bias 7) and 3
  mantissa bits, no infinities, the all-ones exponent-and-mantissa pattern a
  NaN, largest finite value 448 = 1.75 * 2^8, normal numbers down to 2^-6 and
  subnormals m * 2^-9 (m = 1..7).  Encoding rounds to nearest, ties to even,
  and saturates finite values beyond 448 to +-448.
* Q and K are quantised per block: per sequence, per head and per 128-token
  block of that sequence (the kernels' tile), scale = amax / 448 in float32
  (1 for an all-zero block) and code = e4m3(x / scale), the division in
  float32.  Scales are laid out [H, nb]: block kb of sequence b sits at
  column c_b + kb, c_b = b ceil(N / 128) for a dense batch and
  floor(start_b / 128) + b for a packed one; nb is the caller's row stride.
* V is quantised per sequence and head (one scale; the P V product
  accumulates over all key blocks in one accumulator, so one scale per row of
  output), stored transposed as V^T [Hkv, d, vt_tokens]: key j of sequence b at
  column 128 c_b + j, the columns past the sequence up to its next multiple of
  128 zero.
  Scales [Hkv, B].
* Incoherent processing (optional, Q and K only): before the block
  quantisation every row x (d channels) of Q and of K becomes
  R x = (1/sqrt(d)) H_d diag(sigma) x, H_d the Sylvester Hadamard matrix
  (H[i, c] = (-1)^popcount(i & c)) and sigma in {+1, -1}^d drawn from a seed.
  R is orthogonal, so (R q) . (R k) = q . k and the forward needs no change,
  while one large channel is spread over all d (the pages name the technique
  without defining it; this transform is the library's reading).  sigma_c = -1
  where bit c % 32 of word c // 32 of one Philox4x32-10 call (counter
  (0, 2^32 - 1, 2^32 - 1, 0), key (seed mod 2^32, seed // 2^32)) is set.  The
  arithmetic is float32 in a fixed order, so that the codes are reproducible
  bit for bit: the signs (exact), then butterflies (a, b) -> (a + b, a - b) on
  channel pairs (c, c + h), c & h = 0, for h = 1, 2, 4, ..., d/2 in that order,
  each sum rounded to nearest, then one rounded product with float32(1/sqrt(d)).
  The amax, scales and codes are taken from the rotated float32 values.
* The fp8 forward computes, on the dequantised inputs (code value * scale),
  the same O and LSE as the bf16 forward; the kernel rounds the probabilities
  P to e4m3 for the P V product (the row sum uses them unrounded), which
  :func:`o_error_bound` bounds.
"""
from __future__ import annotations

import numpy as np

from . import attention_fwd as _attention_fwd, to_f64
from .dropout import philox4x32_10

E4M3_MAX = 448.0
BLOCK = 128


# ------------------------------------------------------------------ e4m3

def e4m3_decode(codes) -> np.ndarray:
    """uint8 codes -> float64 values (NaN for the two NaN codes)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 0xF) & (m == 0x7), np.nan, mag)
    return sign * mag


def e4m3_encode(x) -> np.ndarray:
    """float values -> uint8 codes: round to nearest, ties to even; finite
    magnitudes beyond 448 saturate to 448; NaN -> 0x7F."""
    x = np.asarray(x, dtype=np.float64)
    sign = np.where(np.signbit(x), 0x80, 0).astype(np.int64)
    a = np.abs(x)
    nan = np.isnan(a)
    a = np.where(nan, 0.0, a)
    # binade exponent of a (exact, from frexp: a = f 2^x with f in [0.5, 1));
    # spacing 2^(e-3) in the normal range, the subnormal spacing 2^-9 below 2^-6
    e = np.frexp(a)[1].astype(np.float64) - 1.0
    e = np.maximum(e, -6.0)
    spacing = np.exp2(e - 3.0)
    q = np.round(a / spacing) * spacing          # np.round: halves to even
    q = np.minimum(q, E4M3_MAX)
    # encode q (exactly representable now)
    normal = q >= 2.0 ** -6
    eq = np.frexp(q)[1].astype(np.float64) - 1.0
    mant = np.where(normal, q / np.exp2(eq) * 8.0 - 8.0, q / 2.0 ** -9)
    code = np.where(normal, ((eq + 7.0).astype(np.int64) << 3) | mant.astype(np.int64),
                    mant.astype(np.int64))
    code = np.where(nan, 0x7F, code | sign)
    return code.astype(np.uint8)


# ------------------------------------------------------------ block layout

def seq_lengths(B: int, N: int, cu_seqlens=None):
    """(start, length) of every sequence."""
    if cu_seqlens is None:
        return [(b * N, N) for b in range(B)]
    cu = [int(c) for c in cu_seqlens]
    return [(cu[b], cu[b + 1] - cu[b]) for b in range(len(cu) - 1)]


def block_offsets(B: int, N: int, cu_seqlens=None):
    """Column c_b of each sequence's first 128-token block in a [H, nb] scale array,
    and the columns the layout spans."""
    seqs = seq_lengths(B, N, cu_seqlens)
    if cu_seqlens is None:
        offs = [b * -(-N // BLOCK) for b in range(B)]
    else:
        offs = [start // BLOCK + b for b, (start, _) in enumerate(seqs)]
    end = max((o + -(-L // BLOCK) for o, (_, L) in zip(offs, seqs)), default=0)
    return offs, end


def vt_offsets(B: int, N: int, cu_seqlens=None):
    """Column of each sequence's first key in the transposed V layout (128 c_b)."""
    offs, end = block_offsets(B, N, cu_seqlens)
    return [BLOCK * o for o in offs], BLOCK * end


def _f32_scale(amax: np.ndarray) -> np.ndarray:
    amax = np.asarray(amax, dtype=np.float32)
    s = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    return np.where(amax > 0, s, np.float32(1.0)).astype(np.float32)


def _encode_scaled(x32: np.ndarray, s32) -> np.ndarray:
    y = (x32 / np.float32(s32)).astype(np.float32)      # float32 division, round to nearest
    return e4m3_encode(y.astype(np.float64))


# --------------------------------------------------- incoherent processing

def hadamard_signs(d: int, seed: int) -> np.ndarray:
    """sigma (float32, +-1) of the rotation for d <= 128 channels: -1 where bit
    c % 32 of word c // 32 of Philox4x32-10 at counter (0, 2^32-1, 2^32-1, 0), key
    (seed mod 2^32, seed // 2^32), is set."""
    assert 0 < d <= 128
    seed = int(seed)
    words = philox4x32_10(0, 0xFFFFFFFF, 0xFFFFFFFF, 0, seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF)
    bits = np.array([(int(words[c // 32]) >> (c % 32)) & 1 for c in range(d)])
    return np.where(bits == 1, np.float32(-1.0), np.float32(1.0)).astype(np.float32)


def rotate(x32: np.ndarray, signs: np.ndarray) -> np.ndarray:
    """R x = (1/sqrt(d)) H_d diag(sigma) x along the last axis, in float32 with the
    library's order of operations: sign flips, then the butterfly stages
    h = 1, 2, ..., d/2 (channel pair (c, c + h) with c & h = 0 becomes
    (a + b, a - b)), then the product with float32(1/sqrt(d))."""
    y = (np.asarray(x32, np.float32) * signs).astype(np.float32)   # exact: sign flips
    d = y.shape[-1]
    lead = y.shape[:-1]
    h = 1
    while h < d:
        # channel c = (g * 2 + half) * h + t: the pairs are (half 0, half 1) of each g
        y = y.reshape(*lead, d // (2 * h), 2, h)
        a, b = y[..., 0, :], y[..., 1, :]
        y = np.stack([a + b, a - b], axis=-2).reshape(*lead, d)   # float32 adds, rounded
        h *= 2
    return (y * np.float32(1.0 / np.sqrt(d))).astype(np.float32)


# --------------------------------------------------------------- quantise

def quantize_qk(x, B: int, N: int, cu_seqlens=None, nb=None, rotate_seed=None):
    """Block quantisation of Q or K in the library layout ([B, N, H, d] or packed
    [T, H, d]; bf16 bit patterns or float).  With ``rotate_seed`` the rows are
    first rotated by :func:`rotate` with ``hadamard_signs(d, rotate_seed)``
    (incoherent processing).  Returns (codes uint8 same shape, scales float32
    [H, nb])."""
    xf = to_f64(x).astype(np.float32)      # bf16 values are exact in float32
    if rotate_seed is not None:
        xf = rotate(xf, hadamard_signs(xf.shape[-1], rotate_seed))
    dense = cu_seqlens is None
    if dense:
        xf = xf.reshape(B * N, *xf.shape[2:])
    H = xf.shape[1]
    offs, total = block_offsets(B, N, cu_seqlens)
    nb = total if nb is None else nb
    codes = np.zeros(xf.shape, np.uint8)
    scales = np.ones((H, nb), np.float32)
    for b, (start, L) in enumerate(seq_lengths(B, N, cu_seqlens)):
        for kb in range(-(-L // BLOCK)):
            r0, r1 = start + kb * BLOCK, start + min(L, (kb + 1) * BLOCK)
            for h in range(H):
                blk = xf[r0:r1, h]
                s = _f32_scale(np.max(np.abs(blk)))
                scales[h, offs[b] + kb] = s
                codes[r0:r1, h] = _encode_scaled(blk, s)
    if dense:
        codes = codes.reshape(B, N, *codes.shape[1:])
    return codes, scales


def quantize_v(v, B: int, N: int, cu_seqlens=None, vt_tokens=None):
    """Quantisation of V: one scale per (sequence, head), codes stored transposed.
    Returns (vt codes uint8 [H, d, vt_tokens], scales float32 [H, B])."""
    vf = to_f64(v).astype(np.float32)
    if cu_seqlens is None:
        vf = vf.reshape(B * N, *vf.shape[2:])
    H, d = vf.shape[1], vf.shape[2]
    offs, total = vt_offsets(B, N, cu_seqlens)
    vt_tokens = total if vt_tokens is None else vt_tokens
    vt = np.zeros((H, d, vt_tokens), np.uint8)
    seqs = seq_lengths(B, N, cu_seqlens)
    scales = np.ones((H, len(seqs)), np.float32)
    for b, (start, L) in enumerate(seqs):
        for h in range(H):
            blk = vf[start:start + L, h]
            # an empty sequence has amax 0 (the max over no magnitudes), so scale 1,
            # as for an all-zero block
            s = _f32_scale(np.max(np.abs(blk)) if blk.size else 0.0)
            scales[h, b] = s
            vt[h, :, offs[b]:offs[b] + L] = _encode_scaled(blk, s).T
    return vt, scales


# ------------------------------------------------------------- dequantise

def dequantize_qk(codes, scales, B: int, N: int, cu_seqlens=None):
    """float64 values in the layout of ``codes``."""
    val = e4m3_decode(codes)
    dense = cu_seqlens is None
    if dense:
        val = val.reshape(B * N, *val.shape[2:])
    offs, _ = block_offsets(B, N, cu_seqlens)
    out = np.zeros_like(val)
    for b, (start, L) in enumerate(seq_lengths(B, N, cu_seqlens)):
        for kb in range(-(-L // BLOCK)):
            r0, r1 = start + kb * BLOCK, start + min(L, (kb + 1) * BLOCK)
            out[r0:r1] = val[r0:r1] * scales[:, offs[b] + kb].astype(np.float64)[None, :, None]
    if dense:
        out = out.reshape(B, N, *out.shape[1:])
    return out


def dequantize_v(vt, scales, B: int, N: int, cu_seqlens=None):
    """float64 V in the library layout ([B, N, H, d] or [T, H, d])."""
    H, d, _ = vt.shape
    seqs = seq_lengths(B, N, cu_seqlens)
    T = seqs[-1][0] + seqs[-1][1]
    offs, _ = vt_offsets(B, N, cu_seqlens)
    out = np.zeros((T, H, d))
    for b, (start, L) in enumerate(seqs):
        blk = e4m3_decode(vt[:, :, offs[b]:offs[b] + L])            # [H, d, L]
        out[start:start + L] = (blk * scales[:, b].astype(np.float64)[:, None, None]).transpose(2, 0, 1)
    if cu_seqlens is None:
        out = out.reshape(B, N, H, d)
    return out


# ---------------------------------------------------------------- forward

def attention_fwd(q8, q_scale, k8, k_scale, vt8, v_scale, *, B: int, N: int, causal: bool,
                  window: int, scale: float, cu_seqlens=None):
    """O and LSE (float64) of exact attention on the dequantised inputs."""
    q = dequantize_qk(q8, q_scale, B, N, cu_seqlens)
    k = dequantize_qk(k8, k_scale, B, N, cu_seqlens)
    v = dequantize_v(vt8, v_scale, B, N, cu_seqlens)
    return _attention_fwd(q, k, v, causal=causal, window=window, scale=scale, cu_seqlens=cu_seqlens)


def o_error_bound(q, k, v, lse, *, causal: bool, window: int, scale: float, rows):
    """Per-element bound on |O_kernel - O| for query rows ``rows`` of one
    (sequence, query head): q [L, d], k, v [L, d] dequantised float64, lse [L].

    The kernel forms p_ij = exp(S_ij - m) for a reference m <= max_j S_ij (so
    every p_ij >= P_ij l_i with P the softmax and l_i >= 1 its normaliser in
    the kernel's units), rounds it to e4m3 for the P V product and divides by
    the unrounded row sum.  Rounding a normal e4m3 value moves it by at most
    2^-4 of itself; a value below 2^-6 (subnormal) by at most 2^-10, and such a
    value has P_ij < 2^-6.  Hence
        |dO_ic| <= 2^-4 sum_j P_ij |V_jc| + 2^-10 sum_{j: P_ij < 2^-6} |V_jc|,
    plus the bf16 rounding of O (2^-8 |O_ic|) and fp32 accumulation (1e-3).
    """
    rows = np.asarray(rows)
    L = k.shape[0]
    s = scale * (q[rows] @ k.T)
    j = np.arange(L)[None, :]
    i = rows[:, None]
    vis = np.broadcast_to(j < L, (len(rows), L)).copy()
    if causal:
        vis &= j <= i
    if window > 0:
        vis &= (i - j) < window
    P = np.where(vis, np.exp(s - lse[rows][:, None]), 0.0)
    av = np.abs(v)
    o = P @ v
    return 2.0 ** -4 * (P @ av) + 2.0 ** -10 * (np.where(vis & (P < 2.0 ** -6), 1.0, 0.0) @ av) \
        + 2.0 ** -8 * np.abs(o) + 1e-3
