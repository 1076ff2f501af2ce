"""The seeded input generators shared by the tests, the benchmark and the oracle
checks (CPU only): bf16 rounding, seed offsets and the packed batch's lengths."""
import numpy as np

from exact_io_aware_tcgen05_gb300 import inputs
from exact_io_aware_tcgen05_gb300.workloads import WORKLOADS


def test_bf16_rounding_ties_to_even():
    # float32 patterns whose low 16 bits are exactly half a bf16 step: the upper half
    # stays when it is even and goes up by one when it is odd
    hi = np.array([0x3F80, 0x3F81, 0xBF80, 0xBF81, 0x4049, 0x404A], np.uint32)
    x = ((hi << 16) | 0x8000).view(np.float32)
    got = inputs.bf16_bits_rne(x)
    want = np.where(hi & 1, hi + 1, hi).astype(np.uint16)
    np.testing.assert_array_equal(got, want)
    # just below and just above the tie go down and up
    np.testing.assert_array_equal(inputs.bf16_bits_rne(((hi << 16) | 0x7FFF).view(np.float32)),
                                  hi.astype(np.uint16))
    np.testing.assert_array_equal(inputs.bf16_bits_rne(((hi << 16) | 0x8001).view(np.float32)),
                                  (hi + 1).astype(np.uint16))


def test_bf16_rounding_is_nearest():
    # every result is a nearest bf16 value of its float32 input
    x = np.random.default_rng(1).standard_normal(20000, dtype=np.float32) * 3
    b = inputs.bf16_bits_rne(x).astype(np.uint32)
    val = (b << 16).view(np.float32).astype(np.float64)
    up = ((b + 1) << 16).view(np.float32).astype(np.float64)
    dn = ((b - 1) << 16).view(np.float32).astype(np.float64)
    err = np.abs(val - x)
    assert np.all(err <= np.abs(up - x)) and np.all(err <= np.abs(dn - x))


def test_seed_offsets_and_reproducibility():
    shape = (2, 9, 3, 8)
    a = inputs.attention_inputs(shape, shape, 5)
    b = inputs.attention_inputs(shape, shape, 5)
    for n in ("q", "k", "v", "dout"):
        np.testing.assert_array_equal(a[n], b[n])
    # Q, K, V, dO draw from seeds s, s + 1, s + 2, s + 3
    for i, n in enumerate(("q", "k", "v", "dout")):
        np.testing.assert_array_equal(a[n], inputs.normal_bf16(shape, 5 + i))


def test_packed_batch_lengths():
    # the packed workloads' 16 lengths, seed 0, uniform on [256, 8192]
    lens = inputs.varlen_lengths(0, 16, 256, 8192)
    assert len(lens) == 16 and lens.min() >= 256 and lens.max() <= 8192
    assert int(lens.sum()) == 68143 and int(lens.max()) == 7960
    w = WORKLOADS["fwdbwd_varlen16_h32kv8_d128_causal"]
    assert list(w.seq_lengths()) == [int(x) for x in lens]
    cu = inputs.cu_seqlens_of(lens)
    assert cu[0] == 0 and cu[-1] == 68143 and np.all(np.diff(cu) == lens)
