"""The C-ABI library on the host (no GPU needed): it loads, exports every symbol
include/fa.h declares, and rejects bad arguments before touching the GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from exact_io_aware_tcgen05_gb300 import build as b
    path = b.build()
    import exact_io_aware_tcgen05_gb300 as fa
    return fa, ctypes.CDLL(path)


def declared_functions():
    names = []
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if f.endswith(".h"):
            text = open(os.path.join(inc, f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w\s\*]*?\b(fa_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("fa_fwd", "fa_bwd", "fa_fwd_typed", "fa_bwd_typed", "fa_fwd_dropout",
              "fa_bwd_dropout", "fa_bwd_workspace_size", "fa_last_error", "fa_device_status",
              "fa_fwd_fp8", "fa_fp8_quantize_qk", "fa_fp8_quantize_v", "fa_fp8_scale_blocks",
              "fa_fp8_vt_tokens", "fa_fp8_quantize_qk_incoherent", "fa_bwd_set_dq_heads",
              "fa_fwd_set_heads"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    _, raw = lib
    missing = [n for n in declared_functions() if not hasattr(raw, n)]
    assert not missing, missing


def _fwd(fa, **over):
    args = dict(q=16, k=16, v=16, o=16, lse=16, B=1, Hq=2, Hkv=1, N=128, d=128, causal=1,
                window=0, cu_seqlens=None, total_tokens=0, scale=0.125)
    args.update(over)
    return fa.fa_fwd(args["q"], args["k"], args["v"], args["o"], args["lse"], args["B"],
                     args["Hq"], args["Hkv"], args["N"], args["d"], args["causal"],
                     args["window"], args["cu_seqlens"], args["total_tokens"], args["scale"],
                     None, check=False)


@pytest.mark.parametrize("over,status", [
    (dict(q=None), 1), (dict(o=8), 1), (dict(d=96), 2), (dict(d=256), 2), (dict(Hkv=3), 1),
    (dict(B=0), 1), (dict(N=0), 1), (dict(window=-1), 1), (dict(window=4, causal=0), 1),
    (dict(scale=0.0), 1), (dict(scale=float("nan")), 1), (dict(scale=-1.0), 1),
    (dict(cu_seqlens=16, total_tokens=-1), 1),
])
def test_forward_rejects_bad_arguments(lib, over, status):
    fa, _ = lib
    assert _fwd(fa, **over) == status
    assert fa.fa_last_error() != ""


def test_typed_entry_points_reject_unknown_element_types(lib):
    fa, _ = lib
    st = fa.fa_fwd_typed(7, 16, 16, 16, 16, 16, 1, 2, 1, 128, 128, 1, 0, None, 0, 0.125, None,
                         check=False)
    assert st == 2 and "element type" in fa.fa_last_error()
    need = fa.fa_bwd_workspace_size(1, 2, 1, 128, 128, 0)
    st = fa.fa_bwd_typed(-1, 16, 16, 16, 16, 16, 16, 16, 16, 16, 1, 2, 1, 128, 128, 1, 0, None, 0,
                         0.125, 256, need, None, check=False)
    assert st == 2 and "element type" in fa.fa_last_error()
    # known element types still get the ordinary argument checks
    st = fa.fa_fwd_typed(fa.FA_DTYPE_F16, None, 16, 16, 16, 16, 1, 2, 1, 128, 128, 1, 0, None, 0,
                         0.125, None, check=False)
    assert st == 1


def test_backward_rejects_small_workspace(lib):
    fa, _ = lib
    need = fa.fa_bwd_workspace_size_min(2, 4, 2, 300, 128, 0)
    st = fa.fa_bwd(16, 16, 16, 16, 16, 16, 16, 16, 16, 2, 4, 2, 300, 128, 1, 0, None, 0, 0.1,
                   256, need - 256, None, check=False)
    assert st == 3 and "workspace" in fa.fa_last_error()
    st = fa.fa_bwd(16, 16, 16, 16, 16, 16, 16, 16, 16, 2, 4, 2, 300, 128, 1, 0, None, 0, 0.1,
                   None, need, None, check=False)
    assert st == 3
    st = fa.fa_bwd(16, 16, 16, 16, 16, 16, 16, 16, 16, 2, 4, 2, 300, 128, 1, 0, None, 0, 0.1,
                   16, need, None, check=False)
    assert st == 3 and "aligned" in fa.fa_last_error()


def _pad(x):
    return (x + 255) // 256 * 256


def test_workspace_size(lib):
    fa, _ = lib
    # split backward: B * Hq * N fp32 row statistics, padded to 256 bytes
    assert fa.fa_bwd_workspace_size_min(2, 16, 16, 8192, 128, 0) == 2 * 16 * 8192 * 4
    assert fa.fa_bwd_workspace_size_min(1, 3, 1, 5, 64, 0) == 256
    # packed: Hq * T
    assert fa.fa_bwd_workspace_size_min(16, 32, 8, 7960, 128, 68143) == _pad(32 * 68143 * 4)
    # fused backward: + fp32 row scales (one per row and head) + the K/V bound slots
    # (32 x (d + 1) fp32 per key/value head) + the int32 dQ sums (d per row and head)
    for B, Hq, Hkv, N, d, T in ((2, 16, 16, 8192, 128, 0), (1, 3, 1, 5, 64, 0),
                                (16, 32, 8, 7960, 128, 68143), (16, 32, 8, 7960, 64, 68143)):
        rows = T if T else B * N
        full = 2 * _pad(rows * Hq * 4) + _pad(Hkv * 32 * (d + 1) * 4) + _pad(rows * Hq * d * 4)
        assert fa.fa_bwd_workspace_size_fused(B, Hq, Hkv, N, d, T) == full
        # the default choice: the fused backward at d = 64, the split one at d = 128
        want = full if d == 64 else fa.fa_bwd_workspace_size_min(B, Hq, Hkv, N, d, T)
        assert fa.fa_bwd_workspace_size(B, Hq, Hkv, N, d, T) == want
    for f in (fa.fa_bwd_workspace_size, fa.fa_bwd_workspace_size_min, fa.fa_bwd_workspace_size_fused):
        assert f(1, 1, 1, 1, 96, 0) == 0


@pytest.mark.parametrize("d", [64, 128])
def test_backward_path_selection(lib, d):
    """Default: the fused backward at d = 64 (any mask) when the workspace holds it,
    the split one otherwise; a thread can force either, and a forced fused call
    without its workspace would fail."""
    fa, _ = lib
    args = (2, 4, 2, 300, d)
    full = fa.fa_bwd_workspace_size_fused(*args, 0)
    least = fa.fa_bwd_workspace_size_min(*args, 0)
    auto_fused = fa.FA_BWD_FUSED if d == 64 else fa.FA_BWD_SPLIT
    try:
        fa.fa_bwd_set_path(fa.FA_BWD_AUTO)
        assert fa.fa_bwd_path(*args, 1, 0, 0, full) == auto_fused
        assert fa.fa_bwd_path(*args, 1, 100, 0, full) == auto_fused
        assert fa.fa_bwd_path(*args, 1, 0, 0, full - 1) == fa.FA_BWD_SPLIT
        assert fa.fa_bwd_path(*args, 0, 0, 0, full) == auto_fused
        assert fa.fa_bwd_path(*args, 0, 0, 0, full - 1) == fa.FA_BWD_SPLIT
        assert fa.fa_bwd_path(*args, 1, 0, 0, least - 1) == -1
        assert fa.fa_bwd_path(2, 4, 2, 300, 96, 1, 0, 0, full) == -1
        fa.fa_bwd_set_path(fa.FA_BWD_SPLIT)
        assert fa.fa_bwd_path(*args, 1, 0, 0, full) == fa.FA_BWD_SPLIT
        fa.fa_bwd_set_path(fa.FA_BWD_FUSED)
        assert fa.fa_bwd_path(*args, 1, 0, 0, full) == fa.FA_BWD_FUSED
        assert fa.fa_bwd_path(*args, 1, 0, 0, full - 1) == -1
        assert fa.fa_bwd_path(*args, 0, 0, 0, full) == fa.FA_BWD_FUSED
        assert fa.fa_bwd_path(*args, 0, 0, 0, full - 1) == -1
        # and fa_bwd itself refuses, before touching the GPU
        st = fa.fa_bwd(16, 16, 16, 16, 16, 16, 16, 16, 16, *args, 1, 0, None, 0, 0.1, 256, least,
                       None, check=False)
        assert st == fa.FA_ERR_WORKSPACE and "fused" in fa.fa_last_error()
    finally:
        fa.fa_bwd_set_path(fa.FA_BWD_AUTO)


def test_dq_heads_knob_is_validated_before_any_launch(lib):
    fa, _ = lib
    with pytest.raises(fa.FAError):
        fa.fa_bwd_set_dq_heads(-1)
    need = fa.fa_bwd_workspace_size(1, 4, 1, 128, 128, 0)
    try:
        fa.fa_bwd_set_path(fa.FA_BWD_SPLIT)
        fa.fa_bwd_set_dq_heads(3)                       # does not divide the group of 4
        assert _bwd(fa, Hq=4, Hkv=1, ws_bytes=need) == fa.FA_ERR_INVALID_ARG
        assert "fa_bwd_set_dq_heads" in fa.fa_last_error()
    finally:
        fa.fa_bwd_set_dq_heads(0)
        fa.fa_bwd_set_path(fa.FA_BWD_AUTO)


def test_fwd_heads_knob_is_validated_before_any_launch(lib):
    fa, _ = lib
    with pytest.raises(fa.FAError):
        fa.fa_fwd_set_heads(-2)
    try:
        fa.fa_fwd_set_heads(3)                          # does not divide the group of 4
        assert _fwd(fa, Hq=4, Hkv=1) == fa.FA_ERR_INVALID_ARG
        assert "fa_fwd_set_heads" in fa.fa_last_error()
    finally:
        fa.fa_fwd_set_heads(0)


def test_heads_per_cta_choices_on_the_measured_workloads(lib):
    """The library's heads-per-CTA choices (with no device to query, the 152 SMs of a
    GB300), each the one measured fastest on GB300: one head per CTA on B2 H16 N8192; two
    per forward CTA on B4 H16 N2048 (short MHA sequences); on the GQA workloads (group of
    4) two per forward CTA and the whole group per dQ CTA at N = 16384 with a 4096-key
    window, and the whole group for both on 16 packed sequences and on 1024 short ones."""
    from exact_io_aware_tcgen05_gb300.workloads import WORKLOADS
    fa, _ = lib
    want = {"fwdbwd_b2_h16_n8192_d128_causal": (1, 1), "fwd_b4_h16_n2048_d128_causal": (2, 1),
            "fwdbwd_b1_h32kv8_n16384_d128_causal_w4096": (2, 4),
            "fwdbwd_varlen16_h32kv8_d128_causal": (4, 4),
            "fwdbwd_varlen1024_h32kv8_d128_causal": (4, 4)}
    for name, (f, q) in want.items():
        w = WORKLOADS[name]
        T = w.total_tokens if w.packed else 0
        args = (w.B, w.Hq, w.Hkv, w.N, w.d, w.causal, w.window, T)
        assert (fa.fa_fwd_heads(*args), fa.fa_bwd_dq_heads(*args)) == (f, q), name


def test_heads_queries_follow_the_thread_knobs(lib):
    """A set count is reported as long as it divides Hq (forward) or the group (dQ);
    otherwise, and for invalid sizes, the queries answer -1 as the calls would fail."""
    fa, _ = lib
    args = (1, 32, 8, 16384, 128, 1, 4096, 0)
    try:
        fa.fa_fwd_set_heads(8)
        fa.fa_bwd_set_dq_heads(2)
        assert fa.fa_fwd_heads(*args) == 8 and fa.fa_bwd_dq_heads(*args) == 2
        fa.fa_fwd_set_heads(3)
        fa.fa_bwd_set_dq_heads(8)                          # divides Hq, not the group of 4
        assert fa.fa_fwd_heads(*args) == -1 and fa.fa_bwd_dq_heads(*args) == -1
    finally:
        fa.fa_fwd_set_heads(0)
        fa.fa_bwd_set_dq_heads(0)
    assert fa.fa_fwd_heads(1, 32, 8, 16384, 96, 1, 0, 0) == -1      # head dimension
    assert fa.fa_bwd_dq_heads(1, 6, 4, 128, 64, 1, 0, 0) == -1       # Hq % Hkv != 0
    assert fa.fa_fwd_heads(1, 32, 8, 16384, 128, 1, 4096, 0) == 2    # knobs were reset


def test_binding_fails_loudly_without_library(tmp_path):
    import exact_io_aware_tcgen05_gb300 as fa
    saved = fa._lib
    try:
        fa._lib = None
        with pytest.raises(RuntimeError):
            fa.load(str(tmp_path / "missing.so"))
    finally:
        fa._lib = saved


def test_dropout_entry_points_reject_bad_probabilities(lib):
    fa, _ = lib
    for p in (-0.1, 1.0, float("nan")):
        st = fa.fa_fwd_dropout(fa.FA_DTYPE_BF16, p, 1, 0, 16, 16, 16, 16, 16, 1, 2, 1, 128, 128,
                               1, 0, None, 0, 0.125, None, check=False)
        assert st == 1 and "p_drop" in fa.fa_last_error()
    st = fa.fa_fwd_dropout(fa.FA_DTYPE_BF16, 0.999, 1, 0, 16, 16, 16, 16, 16, 1, 2, 1, 128, 128,
                           1, 0, None, 0, 0.125, None, check=False)
    assert st == 2
    need = fa.fa_bwd_workspace_size(1, 2, 1, 128, 128, 0)
    st = fa.fa_bwd_dropout(fa.FA_DTYPE_BF16, 1.5, 1, 0, 16, 16, 16, 16, 16, 16, 16, 16, 16, 1, 2, 1,
                           128, 128, 1, 0, None, 0, 0.125, 256, need, None, check=False)
    assert st == 1


def test_fp8_sizes_and_argument_checks(lib):
    fa, _ = lib
    # dense: exact block counts; packed: the column space ceil(T / 128) + B (sequence b
    # starts at column floor(start_b / 128) + b)
    assert fa.fa_fp8_scale_blocks(2, 300, 0, 0) == 6 and fa.fa_fp8_vt_tokens(2, 300, 0, 0) == 768
    assert fa.fa_fp8_scale_blocks(16, 8192, 68143, 1) == 533 + 16
    assert fa.fa_fp8_vt_tokens(16, 8192, 68143, 1) == 128 * (533 + 16)
    assert fa.fa_fp8_scale_blocks(3, 100, 300, 1) == 3 + 3      # lengths 100 each: columns 0, 1, 3
    assert fa.fa_fp8_scale_blocks(0, 100, 0, 0) == 0
    def fwd(**over):
        a = dict(nb=3, vt=384, d=128, N=300, q=16)
        a.update(over)
        return fa.fa_fwd_fp8(a["q"], 16, 16, 16, 16, 16, a["nb"], a["vt"], 16, 16, 1, 1, 1, a["N"],
                             a["d"], 0, 0, None, 0, 0.1, None, check=False)
    assert fwd(d=64) == fa.FA_ERR_UNSUPPORTED
    assert fwd(nb=2) == fa.FA_ERR_INVALID_ARG
    assert fwd(vt=256) == fa.FA_ERR_INVALID_ARG
    assert fwd(vt=400) == fa.FA_ERR_INVALID_ARG                  # not a multiple of 128
    assert fwd(q=None) == fa.FA_ERR_INVALID_ARG
    assert fwd(q=8) == fa.FA_ERR_INVALID_ARG                     # misaligned
    assert fa.fa_fp8_quantize_qk(16, 16, 16, 2, 1, 1, 300, 128, None, 0, None,
                                 check=False) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fp8_quantize_qk(16, 16, 16, 3, 1, 1, 300, 96, None, 0, None,
                                 check=False) == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_fp8_quantize_v(16, 16, 16, 256, 1, 1, 300, 128, None, 0, None,
                                check=False) == fa.FA_ERR_INVALID_ARG
    rot = fa.fa_fp8_quantize_qk_incoherent
    assert rot(16, 16, 16, 2, 1, 1, 300, 128, None, 0, 7, None, check=False) == fa.FA_ERR_INVALID_ARG
    assert rot(16, 16, 16, 3, 1, 1, 300, 96, None, 0, 7, None, check=False) == fa.FA_ERR_UNSUPPORTED
    assert rot(None, 16, 16, 3, 1, 1, 300, 128, None, 0, 7, None,
               check=False) == fa.FA_ERR_INVALID_ARG
    assert rot(16, 8, 16, 3, 1, 1, 300, 128, None, 0, 7, None,
               check=False) == fa.FA_ERR_INVALID_ARG                 # misaligned codes
    assert "fa_fp8_quantize_qk_incoherent" in fa.fa_last_error()


def _bwd(fa, **over):
    need = fa.fa_bwd_workspace_size(1, 2, 1, 128, 128, 0)
    a = dict(q=16, k=16, v=16, o=16, lse=16, dout=16, dq=16, dk=16, dv=16, B=1, Hq=2, Hkv=1,
             N=128, d=128, causal=1, window=0, cu_seqlens=None, total_tokens=0, scale=0.125,
             ws=256, ws_bytes=need)
    a.update(over)
    return fa.fa_bwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["dout"], a["dq"], a["dk"],
                     a["dv"], a["B"], a["Hq"], a["Hkv"], a["N"], a["d"], a["causal"], a["window"],
                     a["cu_seqlens"], a["total_tokens"], a["scale"], a["ws"], a["ws_bytes"], None,
                     check=False)


@pytest.mark.parametrize("over,status", [
    *[(dict(**{n: None}), 1) for n in ("q", "k", "v", "o", "lse", "dout", "dq", "dk", "dv")],
    *[(dict(**{n: 8}), 1) for n in ("q", "k", "v", "o", "dout", "dq", "dk", "dv")],
    (dict(d=96), 2), (dict(Hkv=3), 1), (dict(B=0), 1), (dict(N=0), 1),
    (dict(window=4, causal=0), 1), (dict(scale=0.0), 1),
])
def test_backward_rejects_bad_arguments(lib, over, status):
    """The backward checks every pointer (null, 16-byte alignment), the head grouping,
    the sizes and the mask flags before anything is enqueued, as the forward does."""
    fa, _ = lib
    assert _bwd(fa, **over) == status
    assert fa.fa_last_error() != ""


def test_static_workspace_size_constant_matches_header(lib):
    fa, _ = lib
    text = open(os.path.join(ROOT, "include", "fa.h")).read()
    m = re.search(r"#define\s+FA_STATIC_WORKSPACE_BYTES\s+\((\d+)\s*\*\s*(\d+)\s*\*\s*(\d+)\)", text)
    assert m and int(m[1]) * int(m[2]) * int(m[3]) == fa.FA_STATIC_WORKSPACE_BYTES


def test_rejected_static_workspace_call_uses_up_armed_events(lib):
    """A size the static array cannot hold is rejected before anything is enqueued, and
    the timing events armed for that call are used up with it (as fa_bwd's own argument
    errors do), so they cannot time the thread's next call."""
    fa, _ = lib
    fa.fa_set_launch_events([1])          # one handle: too few for any call, never recorded
    st = fa.fa_bwd_static_workspace(16, 16, 16, 16, 16, 16, 16, 16, 16, 4, 64, 8, 32768, 128,
                                    1, 0, None, 0, 0.1, None, check=False)
    assert st == fa.FA_ERR_WORKSPACE
    # still armed, the next call would fail on the event count; disarmed, it reaches
    # its own argument check
    assert _fwd(fa, q=None) == fa.FA_ERR_INVALID_ARG
    assert "non-null" in fa.fa_last_error()


def test_release_build_has_no_bounds_checks(lib):
    fa, _ = lib
    assert not fa.fa_debug_checks_enabled()
    # refused before any CUDA call
    assert fa.fa_debug_check_selftest(None, check=False) == fa.FA_ERR_UNSUPPORTED
    assert "bounds-checking" in fa.fa_last_error()


def test_bounds_checking_build_exports_the_same_symbols():
    from exact_io_aware_tcgen05_gb300 import build as b
    raw = ctypes.CDLL(b.build(debug=True))
    missing = [n for n in declared_functions() if not hasattr(raw, n)]
    assert not missing, missing
    assert raw.fa_debug_checks_enabled() == 1
