"""Exact IO-aware attention for GB300 (sm_103a): Python binding of libfa_gb300.so.

The functions below carry the names of the C ABI in ``include/fa.h`` and only
marshal arguments: pointers may be given as integers or as objects with a
``data_ptr()`` method (e.g. torch tensors), streams as integers or objects
with a ``cuda_stream`` attribute.  Every step of the computation runs in the
library's CUDA kernels; there is no fallback.  If the compiled library is
missing, :func:`load` raises.

:func:`attention_forward` / :func:`attention_backward` are small conveniences
that allocate the outputs (and the backward workspace) with PyTorch and call
the C ABI.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "FAError", "load", "fa_fwd", "fa_bwd", "fa_fwd_typed", "fa_bwd_typed", "fa_fwd_dropout",
    "fa_bwd_dropout", "fa_bwd_workspace_size", "fa_bwd_workspace_size_min",
    "fa_bwd_workspace_size_fused", "fa_bwd_set_path", "fa_bwd_path", "FA_BWD_AUTO", "FA_BWD_SPLIT",
    "FA_BWD_FUSED",
    "fa_bwd_static_workspace", "FA_STATIC_WORKSPACE_BYTES", "FA_DTYPE_BF16", "FA_DTYPE_F16",
    "fa_fp8_scale_blocks", "fa_fp8_vt_tokens", "fa_fp8_quantize_qk", "fa_fp8_quantize_v",
    "fa_fp8_quantize_qk_incoherent", "fa_bwd_set_dq_heads", "fa_fwd_set_heads", "fa_fwd_heads",
    "fa_bwd_dq_heads",
    "fa_fwd_fp8", "Fp8Operands", "quantize_fp8", "attention_forward_fp8",
    "fa_device_status",
    "fa_set_wait_limit_cycles", "fa_set_launch_events", "fa_last_error", "attention_forward", "attention_backward",
    "fa_debug_checks_enabled", "fa_debug_check_selftest",
    "library_path",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "libfa_gb300.so")

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_WORKSPACE, FA_ERR_CUDA, FA_ERR_TIMEOUT = range(6)
STATUS_NAMES = {0: "FA_OK", 1: "FA_ERR_INVALID_ARG", 2: "FA_ERR_UNSUPPORTED", 3: "FA_ERR_WORKSPACE",
                4: "FA_ERR_CUDA", 5: "FA_ERR_TIMEOUT"}

FA_DTYPE_BF16, FA_DTYPE_F16 = 0, 1   # fa_dtype
FA_STATIC_WORKSPACE_BYTES = 16 * 1024 * 1024   # the array of fa_bwd_static_workspace
FA_BWD_AUTO, FA_BWD_SPLIT, FA_BWD_FUSED = -1, 0, 1   # fa_bwd_path_kind

_lib = None
_vp, _i, _f, _sz, _ll = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_longlong


class FAError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def load(path: str | None = None):
    """Load libfa_gb300.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    # FA_GB300_LIBRARY: another build of the library (e.g. the bounds-checking one)
    path = path or os.environ.get("FA_GB300_LIBRARY") or library_path
    if not os.path.exists(path):
        raise RuntimeError(f"{path} not found: build it with exact_io_aware_tcgen05_gb300.build.build()")
    lib = ctypes.CDLL(path)
    lib.fa_fwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _vp, _i, _f, _vp]
    lib.fa_fwd.restype = _i
    lib.fa_bwd_workspace_size.argtypes = [_i, _i, _i, _i, _i, _i]
    lib.fa_bwd_workspace_size.restype = _sz
    lib.fa_bwd_workspace_size_min.argtypes = [_i, _i, _i, _i, _i, _i]
    lib.fa_bwd_workspace_size_min.restype = _sz
    lib.fa_bwd_workspace_size_fused.argtypes = [_i, _i, _i, _i, _i, _i]
    lib.fa_bwd_workspace_size_fused.restype = _sz
    lib.fa_bwd_set_path.argtypes = [_i]
    lib.fa_bwd_set_path.restype = None
    lib.fa_bwd_set_dq_heads.argtypes = [_i]
    lib.fa_bwd_set_dq_heads.restype = _i
    lib.fa_fwd_set_heads.argtypes = [_i]
    lib.fa_fwd_set_heads.restype = _i
    lib.fa_bwd_path.argtypes = [_i, _i, _i, _i, _i, _i, _i, _i, _sz]
    lib.fa_bwd_path.restype = _i
    for name in ("fa_fwd_heads", "fa_bwd_dq_heads"):
        getattr(lib, name).argtypes = [_i] * 8
        getattr(lib, name).restype = _i
    lib.fa_bwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i,
                           _vp, _i, _f, _vp, _sz, _vp]
    lib.fa_bwd.restype = _i
    lib.fa_fwd_typed.argtypes = [_i] + lib.fa_fwd.argtypes
    lib.fa_fwd_typed.restype = _i
    lib.fa_bwd_typed.argtypes = [_i] + lib.fa_bwd.argtypes
    lib.fa_bwd_typed.restype = _i
    _u64, _u32 = ctypes.c_ulonglong, ctypes.c_uint
    lib.fa_fwd_dropout.argtypes = [_i, _f, _u64, _u32] + lib.fa_fwd.argtypes
    lib.fa_fwd_dropout.restype = _i
    lib.fa_bwd_dropout.argtypes = [_i, _f, _u64, _u32] + lib.fa_bwd.argtypes
    lib.fa_bwd_dropout.restype = _i
    lib.fa_bwd_static_workspace.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i,
                                            _i, _i, _i, _i, _i, _vp, _i, _f, _vp]
    lib.fa_bwd_static_workspace.restype = _i
    lib.fa_fp8_scale_blocks.argtypes = [_i, _i, _i, _i]
    lib.fa_fp8_scale_blocks.restype = _i
    lib.fa_fp8_vt_tokens.argtypes = [_i, _i, _i, _i]
    lib.fa_fp8_vt_tokens.restype = _i
    lib.fa_fp8_quantize_qk.argtypes = [_vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _i, _vp]
    lib.fa_fp8_quantize_qk.restype = _i
    lib.fa_fp8_quantize_qk_incoherent.argtypes = [_vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _i,
                                                  _u64, _vp]
    lib.fa_fp8_quantize_qk_incoherent.restype = _i
    lib.fa_fp8_quantize_v.argtypes = [_vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _i, _vp]
    lib.fa_fp8_quantize_v.restype = _i
    lib.fa_fwd_fp8.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _vp, _vp, _i, _i, _i, _i, _i,
                               _i, _i, _vp, _i, _f, _vp]
    lib.fa_fwd_fp8.restype = _i
    lib.fa_device_status.argtypes = [_vp]
    lib.fa_device_status.restype = _i
    lib.fa_set_wait_limit_cycles.argtypes = [_ll]
    lib.fa_set_wait_limit_cycles.restype = None
    lib.fa_set_launch_events.argtypes = [ctypes.POINTER(ctypes.c_void_p), _i]
    lib.fa_set_launch_events.restype = None
    lib.fa_debug_checks_enabled.argtypes = []
    lib.fa_debug_checks_enabled.restype = _i
    lib.fa_debug_check_selftest.argtypes = [_vp]
    lib.fa_debug_check_selftest.restype = _i
    lib.fa_last_error.argtypes = []
    lib.fa_last_error.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def fa_last_error() -> str:
    return load().fa_last_error().decode()


def _check(st: int):
    if st != FA_OK:
        raise FAError(st, fa_last_error())


def fa_fwd(q, k, v, o, lse, B, Hq, Hkv, N, d, causal, window, cu_seqlens, total_tokens, scale,
           stream=None, check: bool = True) -> int:
    st = load().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, N, d,
                       int(bool(causal)), int(window), _ptr(cu_seqlens), int(total_tokens),
                       float(scale), _stream(stream))
    if check:
        _check(st)
    return st


def fa_bwd_workspace_size(B, Hq, Hkv, N, d, total_tokens) -> int:
    """Workspace bytes of fa_bwd's default choice for this head dimension."""
    return int(load().fa_bwd_workspace_size(B, Hq, Hkv, N, d, int(total_tokens)))


def fa_bwd_workspace_size_min(B, Hq, Hkv, N, d, total_tokens) -> int:
    """The split backward's workspace, the least fa_bwd accepts."""
    return int(load().fa_bwd_workspace_size_min(B, Hq, Hkv, N, d, int(total_tokens)))


def fa_bwd_workspace_size_fused(B, Hq, Hkv, N, d, total_tokens) -> int:
    """The fused backward's workspace."""
    return int(load().fa_bwd_workspace_size_fused(B, Hq, Hkv, N, d, int(total_tokens)))


def fa_bwd_set_path(path) -> None:
    """Backward path of this thread's fa_bwd calls: FA_BWD_AUTO, FA_BWD_SPLIT or FA_BWD_FUSED."""
    load().fa_bwd_set_path(int(path))


def fa_fwd_set_heads(heads: int) -> None:
    """Query heads per forward CTA on this thread (0: automatic; see include/fa.h)."""
    _check(load().fa_fwd_set_heads(int(heads)))


def fa_bwd_set_dq_heads(heads: int) -> None:
    """Query heads per dQ CTA of the split backward on this thread (0: automatic;
    see include/fa.h)."""
    _check(load().fa_bwd_set_dq_heads(int(heads)))


def fa_fwd_heads(B, Hq, Hkv, N, d, causal, window, total_tokens) -> int:
    """Query heads per CTA fa_fwd would serve on this thread for these sizes (total_tokens:
    T for a packed batch, 0 for a dense one; -1: fa_fwd would fail)."""
    return int(load().fa_fwd_heads(B, Hq, Hkv, N, d, int(bool(causal)), int(window),
                                   int(total_tokens)))


def fa_bwd_dq_heads(B, Hq, Hkv, N, d, causal, window, total_tokens) -> int:
    """Query heads per dQ CTA the split backward would serve on this thread (as
    fa_fwd_heads)."""
    return int(load().fa_bwd_dq_heads(B, Hq, Hkv, N, d, int(bool(causal)), int(window),
                                      int(total_tokens)))


def fa_bwd_path(B, Hq, Hkv, N, d, causal, window, total_tokens, workspace_bytes) -> int:
    """FA_BWD_FUSED or FA_BWD_SPLIT: the backward fa_bwd would run on this thread for
    these arguments (-1: it would fail)."""
    return int(load().fa_bwd_path(B, Hq, Hkv, N, d, int(bool(causal)), int(window),
                                  int(total_tokens), int(workspace_bytes)))


def fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, N, d, causal, window, cu_seqlens,
           total_tokens, scale, workspace, workspace_bytes, stream=None, check: bool = True) -> int:
    st = load().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq),
                       _ptr(dk), _ptr(dv), B, Hq, Hkv, N, d, int(bool(causal)), int(window),
                       _ptr(cu_seqlens), int(total_tokens), float(scale), _ptr(workspace),
                       int(workspace_bytes), _stream(stream))
    if check:
        _check(st)
    return st


def fa_fwd_typed(dtype, q, k, v, o, lse, B, Hq, Hkv, N, d, causal, window, cu_seqlens,
                 total_tokens, scale, stream=None, check: bool = True) -> int:
    """fa_fwd for element type ``dtype`` (FA_DTYPE_BF16 or FA_DTYPE_F16)."""
    st = load().fa_fwd_typed(int(dtype), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv,
                             N, d, int(bool(causal)), int(window), _ptr(cu_seqlens),
                             int(total_tokens), float(scale), _stream(stream))
    if check:
        _check(st)
    return st


def fa_bwd_typed(dtype, q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, N, d, causal, window,
                 cu_seqlens, total_tokens, scale, workspace, workspace_bytes, stream=None,
                 check: bool = True) -> int:
    """fa_bwd for element type ``dtype`` (FA_DTYPE_BF16 or FA_DTYPE_F16)."""
    st = load().fa_bwd_typed(int(dtype), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout),
                             _ptr(dq), _ptr(dk), _ptr(dv), B, Hq, Hkv, N, d, int(bool(causal)),
                             int(window), _ptr(cu_seqlens), int(total_tokens), float(scale),
                             _ptr(workspace), int(workspace_bytes), _stream(stream))
    if check:
        _check(st)
    return st


def fa_fwd_dropout(dtype, p_drop, seed, offset, q, k, v, o, lse, B, Hq, Hkv, N, d, causal, window,
                   cu_seqlens, total_tokens, scale, stream=None, check: bool = True) -> int:
    """fa_fwd with dropout of the probabilities (see include/fa.h for the keep mask)."""
    st = load().fa_fwd_dropout(int(dtype), float(p_drop), int(seed), int(offset), _ptr(q), _ptr(k),
                               _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, N, d, int(bool(causal)),
                               int(window), _ptr(cu_seqlens), int(total_tokens), float(scale),
                               _stream(stream))
    if check:
        _check(st)
    return st


def fa_bwd_dropout(dtype, p_drop, seed, offset, q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, N, d,
                   causal, window, cu_seqlens, total_tokens, scale, workspace, workspace_bytes,
                   stream=None, check: bool = True) -> int:
    """fa_bwd of fa_fwd_dropout (same p_drop, seed, offset)."""
    st = load().fa_bwd_dropout(int(dtype), float(p_drop), int(seed), int(offset), _ptr(q), _ptr(k),
                               _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
                               B, Hq, Hkv, N, d, int(bool(causal)), int(window), _ptr(cu_seqlens),
                               int(total_tokens), float(scale), _ptr(workspace),
                               int(workspace_bytes), _stream(stream))
    if check:
        _check(st)
    return st


def fa_bwd_static_workspace(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, N, d, causal, window,
                            cu_seqlens, total_tokens, scale, stream=None, check: bool = True) -> int:
    """fa_bwd without a workspace argument, for callers that cannot allocate device
    memory: the scratch is a fixed array inside the library (FA_STATIC_WORKSPACE_BYTES,
    16 MiB per GPU).  Calls on one device share that array, so calls whose work
    overlaps on the GPU must be serialised."""
    st = load().fa_bwd_static_workspace(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout),
                                        _ptr(dq), _ptr(dk), _ptr(dv), B, Hq, Hkv, N, d,
                                        int(bool(causal)), int(window), _ptr(cu_seqlens),
                                        int(total_tokens), float(scale), _stream(stream))
    if check:
        _check(st)
    return st


def fa_device_status(stream=None, check: bool = True) -> int:
    st = load().fa_device_status(_stream(stream))
    if check:
        _check(st)
    return st


_armed_events = None   # keeps the handle array alive until the armed call has used it


def fa_set_launch_events(events) -> None:
    """Arm per-kernel timing for this thread's next fa_fwd / fa_bwd call.

    ``events``: cudaEvent_t handles (ints) or torch.cuda.Event objects that have
    been recorded at least once; None disarms.
    """
    global _armed_events
    if events is None:
        _armed_events = None
        load().fa_set_launch_events(None, 0)
        return
    handles = [e if isinstance(e, int) else e.cuda_event for e in events]
    _armed_events = (ctypes.c_void_p * len(handles))(*handles)
    load().fa_set_launch_events(_armed_events, len(handles))


def fa_debug_checks_enabled() -> bool:
    """True for the bounds-checking build of the library."""
    return bool(load().fa_debug_checks_enabled())


def fa_debug_check_selftest(stream=None, check: bool = True) -> int:
    st = load().fa_debug_check_selftest(_stream(stream))
    if check:
        _check(st)
    return st


def fa_set_wait_limit_cycles(cycles: int) -> None:
    load().fa_set_wait_limit_cycles(int(cycles))


# ------------------------------------------------------------ conveniences

def fa_fp8_scale_blocks(B, N, total_tokens, packed) -> int:
    """Columns of the fp8 block-scale arrays (see include/fa.h)."""
    return int(load().fa_fp8_scale_blocks(B, N, int(total_tokens), int(bool(packed))))


def fa_fp8_vt_tokens(B, N, total_tokens, packed) -> int:
    """Columns of the transposed fp8 V (see include/fa.h)."""
    return int(load().fa_fp8_vt_tokens(B, N, int(total_tokens), int(bool(packed))))


def fa_fp8_quantize_qk(x, x8, scales, nb, B, H, N, d, cu_seqlens, total_tokens, stream=None,
                       check: bool = True) -> int:
    """bf16 Q or K -> e4m3 codes and per-block scales."""
    st = load().fa_fp8_quantize_qk(_ptr(x), _ptr(x8), _ptr(scales), int(nb), B, H, N, d,
                                   _ptr(cu_seqlens), int(total_tokens), _stream(stream))
    if check:
        _check(st)
    return st


def fa_fp8_quantize_qk_incoherent(x, x8, scales, nb, B, H, N, d, cu_seqlens, total_tokens, seed,
                                  stream=None, check: bool = True) -> int:
    """bf16 Q or K -> rotated (incoherent processing), e4m3 codes and per-block scales."""
    st = load().fa_fp8_quantize_qk_incoherent(_ptr(x), _ptr(x8), _ptr(scales), int(nb), B, H, N, d,
                                              _ptr(cu_seqlens), int(total_tokens),
                                              int(seed) & 0xFFFFFFFFFFFFFFFF, _stream(stream))
    if check:
        _check(st)
    return st


def fa_fp8_quantize_v(v, vt8, scales, vt_tokens, B, H, N, d, cu_seqlens, total_tokens, stream=None,
                      check: bool = True) -> int:
    """bf16 V -> transposed e4m3 codes and per-(sequence, head) scales."""
    st = load().fa_fp8_quantize_v(_ptr(v), _ptr(vt8), _ptr(scales), int(vt_tokens), B, H, N, d,
                                  _ptr(cu_seqlens), int(total_tokens), _stream(stream))
    if check:
        _check(st)
    return st


def fa_fwd_fp8(q8, q_scale, k8, k_scale, vt8, v_scale, nb, vt_tokens, o, lse, B, Hq, Hkv, N, d,
               causal, window, cu_seqlens, total_tokens, scale, stream=None,
               check: bool = True) -> int:
    """The fp8 forward (see include/fa.h)."""
    st = load().fa_fwd_fp8(_ptr(q8), _ptr(q_scale), _ptr(k8), _ptr(k_scale), _ptr(vt8),
                           _ptr(v_scale), int(nb), int(vt_tokens), _ptr(o), _ptr(lse), B, Hq, Hkv,
                           N, d, int(bool(causal)), int(window), _ptr(cu_seqlens),
                           int(total_tokens), float(scale), _stream(stream))
    if check:
        _check(st)
    return st


def _geometry(q, k, cu_seqlens, max_seqlen):
    if cu_seqlens is None:
        B, N, Hq, d = q.shape
        return B, N, Hq, k.shape[2], d, 0
    T, Hq, d = q.shape
    B = cu_seqlens.numel() - 1
    if max_seqlen is None:
        raise ValueError("packed batches need max_seqlen")
    return B, int(max_seqlen), Hq, k.shape[1], d, T


def _dtype_code(*tensors) -> int:
    """fa_dtype of torch tensors that must all be bf16, or all fp16."""
    import torch
    codes = {torch.bfloat16: FA_DTYPE_BF16, torch.float16: FA_DTYPE_F16}
    kinds = {t.dtype for t in tensors}
    if len(kinds) != 1 or next(iter(kinds)) not in codes:
        raise TypeError(f"q, k, v (and o, dout) must all be bfloat16 or all float16, got {kinds}")
    return codes[next(iter(kinds))]


def attention_forward(q, k, v, *, causal=False, window=0, scale=None, cu_seqlens=None,
                      max_seqlen=None, stream=None, dropout=None, heads=0):
    """O, LSE for CUDA tensors q, k, v (all bf16 or all fp16) in the library's layouts
    (allocates outputs).  ``heads``: query heads per CTA for this call (0: the library's
    choice; see fa_fwd_set_heads)."""
    import torch
    dtype = _dtype_code(q, k, v)
    B, N, Hq, Hkv, d, T = _geometry(q, k, cu_seqlens, max_seqlen)
    scale = d ** -0.5 if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty((Hq, T) if cu_seqlens is not None else (B, Hq, N), dtype=torch.float32,
                      device=q.device)
    stream = stream if stream is not None else torch.cuda.current_stream(q.device)
    fa_fwd_set_heads(heads)
    try:
        if dropout is not None:
            p_drop, seed, offset = dropout
            fa_fwd_dropout(dtype, p_drop, seed, offset, q, k, v, o, lse, B, Hq, Hkv, N, d,
                           causal, window, cu_seqlens, T, scale, stream)
        else:
            fa_fwd_typed(dtype, q, k, v, o, lse, B, Hq, Hkv, N, d, causal, window, cu_seqlens,
                         T, scale, stream)
    finally:
        fa_fwd_set_heads(0)
    return o, lse


class Fp8Operands(tuple):
    """(q8, q_scale, k8, k_scale, vt8, v_scale, nb, vt_tokens) of :func:`quantize_fp8`."""
    __slots__ = ()
    _fields = ("q8", "q_scale", "k8", "k_scale", "vt8", "v_scale", "nb", "vt_tokens")

    def __getattr__(self, name):
        return self[self._fields.index(name)]


def quantize_fp8(q, k, v, *, cu_seqlens=None, max_seqlen=None, stream=None,
                 incoherent_seed=None) -> Fp8Operands:
    """e4m3 operands of the fp8 forward from bf16 CUDA tensors q, k, v (allocates them).
    With ``incoherent_seed`` Q and K are rotated by the same random orthogonal matrix
    before the quantisation (incoherent processing; the forward is unchanged)."""
    import torch
    if {q.dtype, k.dtype, v.dtype} != {torch.bfloat16}:
        raise TypeError("quantize_fp8 takes bfloat16 q, k, v")
    B, N, Hq, Hkv, d, T = _geometry(q, k, cu_seqlens, max_seqlen)
    packed = cu_seqlens is not None
    nb = fa_fp8_scale_blocks(B, N, T, packed)
    vt_tokens = fa_fp8_vt_tokens(B, N, T, packed)
    dev = q.device
    q8 = torch.empty(q.shape, dtype=torch.uint8, device=dev)
    k8 = torch.empty(k.shape, dtype=torch.uint8, device=dev)
    vt8 = torch.empty((Hkv, d, vt_tokens), dtype=torch.uint8, device=dev)
    qs = torch.empty((Hq, nb), dtype=torch.float32, device=dev)
    ks = torch.empty((Hkv, nb), dtype=torch.float32, device=dev)
    vs = torch.empty((Hkv, B), dtype=torch.float32, device=dev)
    stream = stream if stream is not None else torch.cuda.current_stream(dev)
    if incoherent_seed is None:
        fa_fp8_quantize_qk(q, q8, qs, nb, B, Hq, N, d, cu_seqlens, T, stream)
        fa_fp8_quantize_qk(k, k8, ks, nb, B, Hkv, N, d, cu_seqlens, T, stream)
    else:
        fa_fp8_quantize_qk_incoherent(q, q8, qs, nb, B, Hq, N, d, cu_seqlens, T, incoherent_seed,
                                      stream)
        fa_fp8_quantize_qk_incoherent(k, k8, ks, nb, B, Hkv, N, d, cu_seqlens, T, incoherent_seed,
                                      stream)
    fa_fp8_quantize_v(v, vt8, vs, vt_tokens, B, Hkv, N, d, cu_seqlens, T, stream)
    return Fp8Operands((q8, qs, k8, ks, vt8, vs, nb, vt_tokens))


def attention_forward_fp8(ops: Fp8Operands, *, causal=False, window=0, scale=None,
                          cu_seqlens=None, max_seqlen=None, stream=None):
    """O (bf16), LSE of the fp8 forward on :func:`quantize_fp8` operands (allocates outputs)."""
    import torch
    q8, qs, k8, ks, vt8, vs, nb, vt_tokens = ops
    B, N, Hq, Hkv, d, T = _geometry(q8, k8, cu_seqlens, max_seqlen)
    scale = d ** -0.5 if scale is None else scale
    o = torch.empty(q8.shape, dtype=torch.bfloat16, device=q8.device)
    lse = torch.empty((Hq, T) if cu_seqlens is not None else (B, Hq, N), dtype=torch.float32,
                      device=q8.device)
    stream = stream if stream is not None else torch.cuda.current_stream(q8.device)
    fa_fwd_fp8(q8, qs, k8, ks, vt8, vs, nb, vt_tokens, o, lse, B, Hq, Hkv, N, d, causal, window,
               cu_seqlens, T, scale, stream)
    return o, lse


_PATHS = {"auto": FA_BWD_AUTO, "split": FA_BWD_SPLIT, "fused": FA_BWD_FUSED}


def attention_backward(q, k, v, o, lse, dout, *, causal=False, window=0, scale=None,
                       cu_seqlens=None, max_seqlen=None, stream=None, workspace=None,
                       dropout=None, path="auto", dq_heads=0):
    """dQ, dK, dV for the forward above (allocates outputs and, if not given, the workspace
    that ``path`` -- "auto", "split" or "fused" -- needs; the path is this thread's
    preference for the call, and so is ``dq_heads``, the split backward's query heads per
    dQ CTA, 0 for the library's choice)."""
    import torch
    dtype = _dtype_code(q, k, v, o, dout)
    B, N, Hq, Hkv, d, T = _geometry(q, k, cu_seqlens, max_seqlen)
    scale = d ** -0.5 if scale is None else scale
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    size = {"auto": fa_bwd_workspace_size, "split": fa_bwd_workspace_size_min,
            "fused": fa_bwd_workspace_size_fused}[path]
    ws_bytes = size(B, Hq, Hkv, N, d, T)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    stream = stream if stream is not None else torch.cuda.current_stream(q.device)
    ws_given = workspace.numel() * workspace.element_size()
    fa_bwd_set_path(_PATHS[path])
    fa_bwd_set_dq_heads(dq_heads)
    try:
        if dropout is not None:
            p_drop, seed, offset = dropout
            fa_bwd_dropout(dtype, p_drop, seed, offset, q, k, v, o, lse, dout, dq, dk, dv, B, Hq,
                           Hkv, N, d, causal, window, cu_seqlens, T, scale, workspace, ws_given,
                           stream)
        else:
            fa_bwd_typed(dtype, q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, N, d, causal,
                         window, cu_seqlens, T, scale, workspace, ws_given, stream)
    finally:
        fa_bwd_set_path(FA_BWD_AUTO)
        fa_bwd_set_dq_heads(0)
    return dq, dk, dv
