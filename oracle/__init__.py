"""fp64 CPU oracle for exact scaled dot-product attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The CUDA library never links, loads or calls it, and this package
imports nothing from the CUDA side.

The arithmetic lives in ``fa_oracle.c`` (plain loops in fp64, OpenMP over
rows).  This module only

* builds that file with gcc into ``oracle/_build/libfa_oracle.so``,
* decodes bf16 bit patterns (uint16) to float64 exactly, and
* slices the library's tensor layouts into the per-(sequence, key/value head)
  arrays the C routines take:

  - dense:  Q, O ``[B, N, Hq, d]``; K, V ``[B, N, Hkv, d]``; LSE ``[B, Hq, N]``
  - packed: Q, O ``[T, Hq, d]``;    K, V ``[T, Hkv, d]``;    LSE ``[Hq, T]``,
    sequence b spanning tokens ``cu_seqlens[b] : cu_seqlens[b+1]``.

Query head h reads key/value head ``h // (Hq // Hkv)`` (consecutive grouping).

What is computed, with sources (page title, then section):
"FlashAttention: How IO-Aware Tiling and Online Softmax Solved Transformer
Memory Bottlenecks" -- "Naive Attention Execution Profile" (S = QK^T,
P = softmax(S), O = PV) and "2. Online Softmax Reduction" (max-subtracted
softmax; the block recurrence, used by :func:`fwd_tiled`);
"Flash Attention -- Fast Memory-Efficient Exact Attention" -- "What Flash
Attention Does" (causal, variable length, GQA/MQA), "Key Features" (sliding
window), "Architecture Overview" (backward from the saved output and
logsumexp).  The backward formulas are the calculus of softmax; the pages give
none.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libfa_oracle.so")
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int)


def build(force: bool = False) -> str:
    """Compile fa_oracle.c with gcc (OpenMP) unless an up-to-date build exists."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.fa_oracle_fwd.argtypes = [_dp, _dp, _dp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, ctypes.c_int, ctypes.c_double, _ip,
                                      ctypes.c_int, _dp, _dp]
        lib.fa_oracle_fwd_tiled.argtypes = [_dp, _dp, _dp, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_double, ctypes.c_int, ctypes.c_int, _dp, _dp]
        lib.fa_oracle_bwd.argtypes = [_dp, _dp, _dp, _dp, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                      _ip, ctypes.c_int, _ip, ctypes.c_int, _dp, _dp, _dp]
        for f in (lib.fa_oracle_fwd, lib.fa_oracle_fwd_tiled, lib.fa_oracle_bwd):
            f.restype = ctypes.c_int
        lib.fa_oracle_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def threads() -> int:
    """OpenMP threads the oracle uses."""
    return int(_load().fa_oracle_threads())


def to_f64(a: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> float64 (exact); float arrays (float16 included)
    are just upcast, also exactly."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def _p(a: np.ndarray):
    return a.ctypes.data_as(_dp)


def _ints(x: Optional[Sequence[int]]):
    if x is None:
        return None, None
    arr = np.ascontiguousarray(np.asarray(x, dtype=np.int32))
    return arr, arr.ctypes.data_as(_ip)


# ---------------------------------------------------------------- per group

def fwd_group(q, k, v, causal: bool, window: int, scale: float, rows=None):
    """One sequence, one key/value head.  q [G, L, d], k/v [L, d] (float64).

    Returns (O [G, n, d], LSE [G, n]) for the requested query rows (all rows
    if ``rows`` is None).
    """
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    G, L, d = q.shape
    rarr, rptr = _ints(rows)
    n = L if rows is None else len(rarr)
    o = np.empty((G, n, d), np.float64)
    lse = np.empty((G, n), np.float64)
    rc = _load().fa_oracle_fwd(_p(q), _p(k), _p(v), G, L, d, int(bool(causal)), int(window),
                               float(scale), rptr, n, _p(o), _p(lse))
    if rc != 0:
        raise ValueError(f"fa_oracle_fwd failed ({rc})")
    return o, lse


def fwd_tiled_group(q, k, v, causal: bool, window: int, scale: float, Br: int, Bc: int):
    """Same as :func:`fwd_group` (all rows) but by the online-softmax block recurrence."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    G, L, d = q.shape
    o = np.empty((G, L, d), np.float64)
    lse = np.empty((G, L), np.float64)
    rc = _load().fa_oracle_fwd_tiled(_p(q), _p(k), _p(v), G, L, d, int(bool(causal)),
                                     int(window), float(scale), int(Br), int(Bc), _p(o), _p(lse))
    if rc != 0:
        raise ValueError(f"fa_oracle_fwd_tiled failed ({rc})")
    return o, lse


def bwd_group(q, k, v, dout, causal: bool, window: int, scale: float, qrows=None, krows=None):
    """One sequence, one key/value head.  Returns (dQ [G, nq, d], dK [nk, d], dV [nk, d])."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    dout = np.ascontiguousarray(dout, dtype=np.float64)
    G, L, d = q.shape
    qa, qp = _ints(qrows)
    ka, kp = _ints(krows)
    nq = L if qrows is None else len(qa)
    nk = L if krows is None else len(ka)
    dq = np.empty((G, nq, d), np.float64)
    dk = np.empty((nk, d), np.float64)
    dv = np.empty((nk, d), np.float64)
    rc = _load().fa_oracle_bwd(_p(q), _p(k), _p(v), _p(dout), G, L, d, int(bool(causal)),
                               int(window), float(scale), qp, nq, kp, nk, _p(dq), _p(dk), _p(dv))
    if rc != 0:
        raise ValueError(f"fa_oracle_bwd failed ({rc})")
    return dq, dk, dv


# ------------------------------------------------------------ layout helpers

def _sequences(q, cu_seqlens):
    """Yield (b, token slice) per sequence for the dense or packed layout."""
    if cu_seqlens is None:
        B, N = q.shape[0], q.shape[1]
        for b in range(B):
            yield b, (b, slice(0, N))
    else:
        cu = np.asarray(cu_seqlens, dtype=np.int64)
        for b in range(len(cu) - 1):
            yield b, (None, slice(int(cu[b]), int(cu[b + 1])))


def _take(x, sel):
    b, sl = sel
    return x[b, sl] if b is not None else x[sl]


def _lse_shape(q, Hq, cu_seqlens):
    if cu_seqlens is None:
        return (q.shape[0], Hq, q.shape[1])
    return (Hq, q.shape[0])


def attention_fwd(q, k, v, *, causal: bool = False, window: int = 0, scale: float,
                  cu_seqlens=None):
    """Full forward in the library's layouts.  Returns (O float64, LSE float64)."""
    q, k, v = to_f64(q), to_f64(k), to_f64(v)
    Hq, Hkv = q.shape[-2], k.shape[-2]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    G = Hq // Hkv
    o = np.zeros(q.shape, np.float64)
    lse = np.full(_lse_shape(q, Hq, cu_seqlens), -np.inf)
    for b, sel in _sequences(q, cu_seqlens):
        qs, ks, vs = _take(q, sel), _take(k, sel), _take(v, sel)   # [L, H, d]
        for g in range(Hkv):
            og, lg = fwd_group(qs[:, g * G:(g + 1) * G].transpose(1, 0, 2), ks[:, g], vs[:, g],
                               causal, window, scale)
            if sel[0] is not None:
                o[b, sel[1], g * G:(g + 1) * G] = og.transpose(1, 0, 2)
                lse[b, g * G:(g + 1) * G, sel[1]] = lg
            else:
                o[sel[1], g * G:(g + 1) * G] = og.transpose(1, 0, 2)
                lse[g * G:(g + 1) * G, sel[1]] = lg
    return o, lse


def attention_bwd(q, k, v, dout, *, causal: bool = False, window: int = 0, scale: float,
                  cu_seqlens=None):
    """Full backward in the library's layouts.  Returns (dQ, dK, dV) in float64."""
    q, k, v, dout = to_f64(q), to_f64(k), to_f64(v), to_f64(dout)
    Hq, Hkv = q.shape[-2], k.shape[-2]
    G = Hq // Hkv
    dq = np.zeros(q.shape, np.float64)
    dk = np.zeros(k.shape, np.float64)
    dv = np.zeros(v.shape, np.float64)
    for b, sel in _sequences(q, cu_seqlens):
        qs, ks, vs, ds = _take(q, sel), _take(k, sel), _take(v, sel), _take(dout, sel)
        for g in range(Hkv):
            hs = slice(g * G, (g + 1) * G)
            dqg, dkg, dvg = bwd_group(qs[:, hs].transpose(1, 0, 2), ks[:, g], vs[:, g],
                                      ds[:, hs].transpose(1, 0, 2), causal, window, scale)
            if sel[0] is not None:
                dq[b, sel[1], hs] = dqg.transpose(1, 0, 2)
                dk[b, sel[1], g] = dkg
                dv[b, sel[1], g] = dvg
            else:
                dq[sel[1], hs] = dqg.transpose(1, 0, 2)
                dk[sel[1], g] = dkg
                dv[sel[1], g] = dvg
    return dq, dk, dv


def sequence_views(x, b, cu_seqlens, heads=None):
    """[L, H, d] array of sequence b in either layout (float64), optionally only the
    heads in the slice ``heads``.  Only the selected part is decoded."""
    if cu_seqlens is None:
        part = x[b]
    else:
        cu = np.asarray(cu_seqlens, dtype=np.int64)
        part = x[int(cu[b]):int(cu[b + 1])]
    if heads is not None:
        part = part[:, heads]
    return to_f64(part)


def fwd_rows(q, k, v, b: int, h: int, rows, *, causal: bool, window: int, scale: float,
             cu_seqlens=None):
    """O rows [n, d] and LSE [n] of query head h of sequence b, for the given rows only."""
    Hq, Hkv = q.shape[-2], k.shape[-2]
    G = Hq // Hkv
    g = h // G
    qs = sequence_views(q, b, cu_seqlens, slice(h, h + 1)).transpose(1, 0, 2)
    ks = sequence_views(k, b, cu_seqlens, g)
    vs = sequence_views(v, b, cu_seqlens, g)
    o, lse = fwd_group(qs, ks, vs, causal, window, scale, rows=rows)
    return o[0], lse[0]


def bwd_rows(q, k, v, dout, b: int, g: int, qrows, krows, *, causal: bool, window: int,
             scale: float, cu_seqlens=None):
    """dQ [G, nq, d] for the group's query heads at qrows; dK, dV [nk, d] at krows."""
    Hq, Hkv = q.shape[-2], k.shape[-2]
    G = Hq // Hkv
    hs = slice(g * G, (g + 1) * G)
    qs = sequence_views(q, b, cu_seqlens, hs).transpose(1, 0, 2)
    ds = sequence_views(dout, b, cu_seqlens, hs).transpose(1, 0, 2)
    ks = sequence_views(k, b, cu_seqlens, g)
    vs = sequence_views(v, b, cu_seqlens, g)
    return bwd_group(qs, ks, vs, ds, causal, window, scale, qrows=qrows, krows=krows)
