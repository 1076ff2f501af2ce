"""The attention workloads this library is measured and checked on, and their FLOP counts.

Each workload is named by what it is and its sizes.  FLOPs are algorithmic:
only visible (query, key) pairs count.  The forward pass counts 4*d per pair
and query head (S = QK^T and O = PV, 2*d each).  The backward pass counts
10*d: the five products a backward pass needs (S recomputed once, dP, dV, dK
and dQ), i.e. the customary 2.5x the forward.  Extra products a kernel
issues beyond those (a second S and dP for a split dQ pass) are not counted,
nor is masked-out work.  Causal masking therefore halves the count, and a
sliding window of W keys counts sum_i min(i + 1, W).
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Optional, Tuple

from .inputs import cu_seqlens_of, varlen_lengths


@dataclass(frozen=True)
class Workload:
    name: str
    B: int                 # sequences in the batch
    Hq: int                # query heads
    Hkv: int               # key/value heads (Hq % Hkv == 0)
    N: int                 # sequence length (packed: the longest sequence)
    d: int                 # head dimension
    causal: bool
    window: int            # 0: none; else keys visible per query, including itself
    backward: bool         # whether the workload includes the backward pass
    lengths: Optional[Tuple[int, ...]] = None   # packed batch: per-sequence lengths
    dtype: str = "bf16"    # element type of the 16-bit tensors: "bf16" or "f16"; "fp8": the
                           # fp8 forward on e4m3 operands quantised from bf16 inputs
    p_drop: float = 0.0    # dropout probability of the attention probabilities (0: none)
    incoherent: bool = False   # fp8: rotate Q and K before quantising (incoherent processing)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def packed(self) -> bool:
        return self.lengths is not None

    @property
    def total_tokens(self) -> int:
        return int(sum(self.lengths)) if self.packed else self.B * self.N

    def cu_seqlens(self):
        return cu_seqlens_of(self.lengths) if self.packed else None

    @property
    def q_shape(self):
        return (self.total_tokens, self.Hq, self.d) if self.packed else (self.B, self.N, self.Hq, self.d)

    @property
    def kv_shape(self):
        return (self.total_tokens, self.Hkv, self.d) if self.packed else (self.B, self.N, self.Hkv, self.d)

    @property
    def lse_shape(self):
        return (self.Hq, self.total_tokens) if self.packed else (self.B, self.Hq, self.N)

    def seq_lengths(self):
        return list(self.lengths) if self.packed else [self.N] * self.B

    def visible_pairs_per_head(self) -> int:
        return sum(visible_pairs(L, self.causal, self.window) for L in self.seq_lengths())

    def fwd_flops(self) -> int:
        return 4 * self.d * self.Hq * self.visible_pairs_per_head()

    def bwd_flops(self) -> int:
        return 10 * self.d * self.Hq * self.visible_pairs_per_head()

    def fwd_io_bytes(self) -> int:
        """Algorithmic HBM bytes of one forward: read Q, K, V; write O and LSE once
        (fp8: one-byte Q, K, V, two-byte O)."""
        T = self.total_tokens
        if self.dtype == "fp8":
            return T * self.d * (self.Hq + 2 * self.Hkv) + 2 * T * self.d * self.Hq + 4 * T * self.Hq
        return 2 * T * self.d * (2 * self.Hq + 2 * self.Hkv) + 4 * T * self.Hq

    def bwd_io_bytes(self) -> int:
        """Algorithmic HBM bytes of one backward: read Q, K, V, O, dO, LSE; write dQ, dK, dV."""
        T = self.total_tokens
        return (2 * T * self.d * (3 * self.Hq + 2 * self.Hkv)      # Q, O, dO, K, V
                + 4 * T * self.Hq                                     # LSE
                + 2 * T * self.d * (self.Hq + 2 * self.Hkv))          # dQ, dK, dV

    def kernel_io_bytes(self, kernel: str, fused: bool = False) -> int:
        """Algorithmic HBM bytes of one launch of a library kernel: each tensor the kernel
        must read or write, once (16-bit Q, K, V, O, dO and gradients; fp32 LSE, D and row
        scales; the fused backward's int32 dQ sums).  ``fused``: the preprocess of the
        fused backward, which also writes the row scales, zeroes the dQ sums and reads K
        and V for their bounds."""
        T, d = self.total_tokens, self.d
        q, kv, rows = T * self.Hq * d, T * self.Hkv * d, T * self.Hq
        e = 2
        if kernel == "fa_fwd":
            return self.fwd_io_bytes()
        if kernel == "fa_bwd_preprocess":            # O, dO in; D out
            return 2 * e * q + 4 * rows + ((4 * rows + 4 * q + 2 * e * kv) if fused else 0)
        if kernel == "fa_bwd_dkdv":                  # Q, dO, K, V, LSE, D in; dK, dV out
            return e * (2 * q + 2 * kv) + 8 * rows + 2 * e * kv
        if kernel == "fa_bwd_dq":                    # Q, dO, K, V, LSE, D in; dQ out
            return e * (2 * q + 2 * kv) + 8 * rows + e * q
        if kernel == "fa_bwd_fused":                 # + row scales in; dK, dV, int32 dQ sums out
            return e * (2 * q + 2 * kv) + 12 * rows + 2 * e * kv + 4 * q
        if kernel == "fa_bwd_dq_convert":            # int32 sums and row scales in, dQ out
            return 4 * q + 4 * rows + e * q
        raise KeyError(kernel)


def visible_pairs(L: int, causal: bool, window: int) -> int:
    """Number of (query, key) pairs with key visible to query in one sequence of length L."""
    if not causal:
        return L * L
    if window <= 0 or window >= L:
        return L * (L + 1) // 2
    return window * (window + 1) // 2 + (L - window) * window


def _varlen(d: int) -> Workload:
    lengths = tuple(int(x) for x in varlen_lengths(0, 16, 256, 8192))
    return Workload(f"fwdbwd_varlen16_h32kv8_d{d}_causal", B=len(lengths), Hq=32, Hkv=8,
                    N=max(lengths), d=d, causal=True, window=0, backward=True, lengths=lengths)


def _many_short() -> Workload:
    # a packed batch of many short sequences: 1024 lengths drawn uniformly from [64, 512]
    lengths = tuple(int(x) for x in varlen_lengths(0, 1024, 64, 512))
    return Workload("fwdbwd_varlen1024_h32kv8_d128_causal", B=len(lengths), Hq=32, Hkv=8,
                    N=max(lengths), d=128, causal=True, window=0, backward=True, lengths=lengths)


WORKLOADS = {
    w.name: w for w in [
        Workload("fwd_b1_h1_n128_d64", 1, 1, 1, 128, 64, False, 0, False),
        Workload("fwd_b4_h16_n2048_d128_causal", 4, 16, 16, 2048, 128, True, 0, False),
        Workload("fwdbwd_b2_h16_n8192_d128_causal", 2, 16, 16, 8192, 128, True, 0, True),
        Workload("fwdbwd_b1_h32kv8_n16384_d128_causal_w4096", 1, 32, 8, 16384, 128, True, 4096,
                 True),
        Workload("fwdbwd_b2_h16_n8192_d128_causal_f16", 2, 16, 16, 8192, 128, True, 0, True,
                 dtype="f16"),
        Workload("fwdbwd_b2_h16_n8192_d128_causal_dropout10", 2, 16, 16, 8192, 128, True, 0, True,
                 p_drop=0.1),
        Workload("fwd_b2_h16_n8192_d128_causal_fp8", 2, 16, 16, 8192, 128, True, 0, False,
                 dtype="fp8"),
        Workload("fwd_b2_h16_n8192_d128_causal_fp8_incoherent", 2, 16, 16, 8192, 128, True, 0,
                 False, dtype="fp8", incoherent=True),
        _varlen(128),
        _varlen(64),
        _many_short(),
        # without a causal mask: 8 x 2048 tokens, 32 heads of 64 channels (width 2048)
        Workload("fwdbwd_b8_h32_n2048_d64", 8, 32, 32, 2048, 64, False, 0, True),
    ]
}

#: dropout seed and offset of the workloads with p_drop > 0
DROPOUT_SEED, DROPOUT_OFFSET = 0x5EED, 0

#: rotation seed of the fp8 workloads with incoherent processing
INCOHERENT_SEED = 0x1C0

#: the workload the benchmark times by default: long causal sequences, d = 128, fwd + bwd
BENCH_DEFAULT = "fwdbwd_b2_h16_n8192_d128_causal"
