"""Named synthetic workloads of the TP-MLP block (shapes and value distributions).

Each workload is a transformer MLP of hidden size h and ffn size F = 4h applied to
T = b*s tokens, split into t tensor-parallel shards, the way the "Megatron-LM"
industry report (section 4.1) splits the MLP and the paper's notes size it
(tensor parallelism up to 8 ways inside a server).  Values are Gaussian with the
standard deviations below; a std of 0 gives an all-zero tensor (still drawn, so
the draw order never changes).
"""
from __future__ import annotations

import dataclasses
import math


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    tokens: int
    hidden: int
    ffn: int
    shards: tuple          # the shard counts t this workload is run with
    dtype: str             # "f32" or "bf16": dtype of every input and output
    std_X: float = 1.0
    std_A: float = 0.02
    std_a: float = 0.0
    std_B: float = 0.02
    std_b: float = 0.0
    std_dZ: float = 1.0
    note: str = ""

    @property
    def flops_fwd(self) -> float:
        """Two GEMMs of 2*T*h*F each (bias, GeLU and column sums not counted)."""
        return 4.0 * self.tokens * self.hidden * self.ffn

    @property
    def flops_fwd_bwd(self) -> float:
        """Forward plus backward: three times the forward GEMM work."""
        return 3.0 * self.flops_fwd

    def with_tokens(self, tokens: int) -> "Workload":
        return dataclasses.replace(self, tokens=tokens)


def _sweep(b: int) -> Workload:
    return Workload(f"h12288-b{b}", 2048 * b, 12288, 49152, (8,), "bf16",
                    note="microbatch sweep, s=2048, b=%d" % b)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny-fp32", 128, 256, 1024, (2,), "f32", std_a=0.01, std_b=0.01,
                 note="b=2, s=64; fp32 end to end"),
        Workload("h2048", 2048, 2048, 8192, (1, 2, 4), "bf16", note="b=1, s=2048"),
        Workload("h4096", 8192, 4096, 16384, (8,), "bf16", note="b=4, s=2048"),
        Workload("h8192", 4096, 8192, 32768, (8,), "bf16",
                 std_B=0.02 / math.sqrt(2 * 96),
                 note="b=2, s=2048; B scaled by 1/sqrt(2*96 layers)"),
        _sweep(1), _sweep(2), _sweep(4), _sweep(8),
    ]
}

# The workload the headline throughput is measured on.
HEADLINE = "h8192"


@dataclasses.dataclass(frozen=True)
class AttnWorkload:
    """Causal self-attention over `batch` sequences of `seq` tokens, hidden size
    h, `heads` heads of d = h/heads, split into t shards by heads (the
    "Megatron-LM" industry report, section 4.1)."""
    name: str
    batch: int
    seq: int
    hidden: int
    heads: int
    t: int
    std_X: float = 1.0
    std_W: float = 0.02
    std_b: float = 0.0
    std_dZ: float = 1.0
    note: str = ""

    @property
    def tokens(self) -> int:
        return self.batch * self.seq

    @property
    def flops_fwd(self) -> float:
        """QKV and output projections (2*T*h*3h + 2*T*h*h) plus the two per-head
        products Q K^T and P V over the causal lower triangle only: per head
        seq*(seq+1)/2 dot products of length d each, 2*T*h*(seq+1) for both.
        The masked upper triangle is not counted (the kernels skip it)."""
        T, h = self.tokens, self.hidden
        return 8.0 * T * h * h + 2.0 * T * h * (self.seq + 1)

    @property
    def flops_fwd_bwd(self) -> float:
        """Backward: dO, dWo, dWqkv, dX (twice the projections) and dV, dP, dQ, dK
        (twice the per-head products): three times the forward in total."""
        return 3.0 * self.flops_fwd


ATTN_WORKLOADS = {
    w.name: w
    for w in [
        AttnWorkload("attn-h4096", 4, 2048, 4096, 32, 8, note="b=4, s=2048, d=128"),
        AttnWorkload("attn-h8192", 2, 2048, 8192, 64, 8, note="b=2, s=2048, d=128"),
    ]
}
