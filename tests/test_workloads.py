"""The algorithmic FLOP counts every TFLOP/s figure rests on (CPU only).

workloads.visible_pairs gives the number of (query, key) pairs a sequence's mask
lets through, in closed form.  Here it is checked against a direct count of the
mask's definition: key j is visible to query i iff j <= i (causal) and i - j <
window (window > 0), in one sequence; on small lengths pair by pair, and on every
benchmarked workload's own lengths with a vectorised count.
"""
import numpy as np
import pytest

from exact_io_aware_tcgen05_gb300.workloads import WORKLOADS, visible_pairs


def count_visible(L: int, causal: bool, window: int) -> int:
    total = 0
    j = np.arange(L)
    for i0 in range(0, L, 1024):
        i = np.arange(i0, min(L, i0 + 1024))[:, None]
        vis = np.ones((i.shape[0], L), bool)
        if causal:
            vis &= j[None, :] <= i
        if window > 0:
            vis &= (i - j[None, :]) < window
        total += int(vis.sum())
    return total


@pytest.mark.parametrize("causal", [False, True])
def test_visible_pairs_against_the_mask_pair_by_pair(causal):
    for L in list(range(1, 41)) + [127, 128, 129, 300]:
        for window in (0, 1, 2, 5, L - 1, L, L + 3):
            if window > 0 and not causal:
                continue        # a window needs the causal mask (rejected by the library)
            want = sum(1 for i in range(L) for jj in range(L)
                       if (not causal or jj <= i) and (window <= 0 or i - jj < window))
            assert visible_pairs(L, causal, window) == want, (L, causal, window)


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_workload_pairs_and_flops(name):
    w = WORKLOADS[name]
    pairs = sum(count_visible(L, w.causal, w.window) for L in w.seq_lengths())
    assert w.visible_pairs_per_head() == pairs
    # forward: S = Q K^T and O = P V, 2 d FLOPs per visible pair each; backward: the
    # five products S, dP, dV, dK, dQ (the dQ kernel's recomputed S and dP not counted)
    assert w.fwd_flops() == 4 * w.d * w.Hq * pairs
    assert w.bwd_flops() == 10 * w.d * w.Hq * pairs


def test_closed_forms_of_the_dense_workloads():
    # causal N(N+1)/2; causal with window W < N: W(W+1)/2 + (N - W) W
    assert WORKLOADS["fwdbwd_b2_h16_n8192_d128_causal"].visible_pairs_per_head() == 2 * 8192 * 8193 // 2
    assert WORKLOADS["fwdbwd_b1_h32kv8_n16384_d128_causal_w4096"].visible_pairs_per_head() == \
        4096 * 4097 // 2 + (16384 - 4096) * 4096
    assert WORKLOADS["fwd_b1_h1_n128_d64"].visible_pairs_per_head() == 128 * 128
    assert WORKLOADS["fwdbwd_b8_h32_n2048_d64"].visible_pairs_per_head() == 8 * 2048 * 2048


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_io_bytes_are_the_tensors_read_and_written_once(name):
    """The algorithmic HBM bytes equal the sizes of the tensors each pass reads and
    writes once, taken from their shapes: the forward reads Q, K, V and writes O and
    LSE; the backward reads Q, K, V, O, dO and LSE and writes dQ, dK and dV."""
    w = WORKLOADS[name]
    n = lambda shape: int(np.prod(shape))
    q, kv, lse = n(w.q_shape), n(w.kv_shape), n(w.lse_shape)
    if w.dtype == "fp8":
        assert w.fwd_io_bytes() == 1 * (q + 2 * kv) + 2 * q + 4 * lse
    else:
        assert w.fwd_io_bytes() == 2 * (q + 2 * kv) + 2 * q + 4 * lse
        assert w.bwd_io_bytes() == 2 * (3 * q + 2 * kv) + 4 * lse + 2 * (q + 2 * kv)


def test_kernel_flop_credits_add_up():
    """The kernels' credited FLOPs per pair and unit of d add up to the step's
    algorithmic count on both backward paths (forward 4, backward 10), and the executed
    count differs only for the dQ kernel, which also rebuilds S and dP (3 products)."""
    import bench
    cr, ex = bench.KERNEL_FLOPS_PER_PAIR_D, bench.KERNEL_EXECUTED_FLOPS_PER_PAIR_D
    assert cr["fa_fwd"] == 4
    assert cr["fa_bwd_dkdv"] + cr["fa_bwd_dq"] == 10 and cr["fa_bwd_fused"] == 10
    assert set(cr) == set(ex)
    assert {k for k in cr if cr[k] != ex[k]} == {"fa_bwd_dq"}
    assert ex["fa_bwd_dq"] == 3 * 2


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_kernel_io_bytes_are_the_tensors_each_kernel_moves(name):
    """Per-kernel algorithmic bytes, from the tensor shapes: the dK/dV and dQ kernels
    each read Q, dO, K, V, LSE and D and write their own gradients; the fused backward
    writes dK, dV and the int32 dQ sums; the preprocess reads O and dO and writes D."""
    w = WORKLOADS[name]
    n = lambda shape: int(np.prod(shape))
    q, kv, rows = n(w.q_shape), n(w.kv_shape), n(w.lse_shape)
    assert w.kernel_io_bytes("fa_fwd") == w.fwd_io_bytes()
    reads = 2 * (2 * q + 2 * kv) + 4 * rows + 4 * rows
    assert w.kernel_io_bytes("fa_bwd_dkdv") == reads + 2 * (2 * kv)
    assert w.kernel_io_bytes("fa_bwd_dq") == reads + 2 * q
    assert w.kernel_io_bytes("fa_bwd_fused") == reads + 4 * rows + 2 * (2 * kv) + 4 * q
    assert w.kernel_io_bytes("fa_bwd_preprocess") == 2 * 2 * q + 4 * rows
    assert w.kernel_io_bytes("fa_bwd_dq_convert") == 4 * q + 4 * rows + 2 * q


def test_roofline_bound_follows_arithmetic_intensity():
    """The kernels of the long-sequence workloads are tensor-bound at the measured peaks
    (1875 TFLOP/s, 6788 GB/s: a ridge near 276 FLOP/B); those of 1024 sequences of
    64-512 tokens and the single 128-token tile are HBM-bound."""
    import bench
    def bound(name, kernel):
        w = WORKLOADS[name]
        fl = bench.KERNEL_FLOPS_PER_PAIR_D[kernel] * w.d * w.visible_pairs_per_head() * w.Hq
        return bench.binding_roof(fl / 1e12, w.kernel_io_bytes(kernel), 1875.4, 6788.3)
    # the rule itself: equal times go to the tensor roof
    assert bench.binding_roof(1.0, 1e9 * 6788.3 / 1875.4, 1875.4, 6788.3) == "tensor"
    assert bench.binding_roof(1.0, 1.01e9 * 6788.3 / 1875.4, 1875.4, 6788.3) == "hbm"
    for k in ("fa_fwd", "fa_bwd_dkdv", "fa_bwd_dq", "fa_bwd_fused"):
        assert bound("fwdbwd_b2_h16_n8192_d128_causal", k) == "tensor"
        assert bound("fwdbwd_varlen1024_h32kv8_d128_causal", k) == "hbm"
    assert bound("fwd_b4_h16_n2048_d128_causal", "fa_fwd") == "tensor"
    assert bound("fwd_b1_h1_n128_d64", "fa_fwd") == "hbm"


def test_bench_reports_the_heads_the_kernels_serve():
    """The bench line's heads per CTA: the library's choice for 16-bit calls without
    dropout, one for dropout and fp8 forwards, and no dQ count without a split backward."""
    import bench
    assert bench.served_heads(WORKLOADS["fwdbwd_b1_h32kv8_n16384_d128_causal_w4096"], False, True, False) == (2, 4)
    assert bench.served_heads(WORKLOADS["fwdbwd_b2_h16_n8192_d128_causal_dropout10"], False, True, False) == (1, 1)
    assert bench.served_heads(WORKLOADS["fwd_b2_h16_n8192_d128_causal_fp8"], True, False, False) == (1, None)
    assert bench.served_heads(WORKLOADS["fwdbwd_varlen16_h32kv8_d64_causal"], False, True, True) == (4, None)


def test_traffic_records_follow_the_kernel_sources(tmp_path, monkeypatch):
    """bench.py reports a kernel's recorded DRAM bytes only while the hash of its source
    files (which exist, one entry per kernel) is the one stored with the record."""
    import json
    import os
    import bench
    csrc = os.path.join(bench.ROOT, "exact_io_aware_tcgen05_gb300", "csrc")
    kernels = set(bench.KERNEL_FLOPS_PER_PAIR_D) | {"fa_bwd_preprocess", "fa_bwd_dq_convert"}
    assert set(bench.KERNEL_SOURCES) == kernels
    for k, files in bench.KERNEL_SOURCES.items():
        for f in files + tuple(bench.SHARED_SOURCES):
            assert os.path.exists(os.path.join(csrc, f)), (k, f)
        assert len(bench.source_sha(k)) == 16
    (tmp_path / "profiles").mkdir()
    rec = {"about": "test", "w": {"fa_fwd": {"dram_bytes_per_launch": 123, "source_sha": "a" * 16},
                                  "fa_bwd_dkdv": {"dram_bytes_per_launch": 456, "source_sha": "b" * 16}}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_sha", lambda k: "a" * 16)
    assert bench.recorded_traffic("fa_fwd", "w") == 123
    assert bench.recorded_traffic("fa_bwd_dkdv", "w") is None      # source changed since
    assert bench.recorded_traffic("fa_fwd", "other") is None        # never captured
