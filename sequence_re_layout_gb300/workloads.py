"""Named attention-activation shapes used by the parity tests and the bench.

Model names are shape labels only (head counts and head dimension of their
attention layers); no weights or data are involved.  Each entry gives
``(B, S, Hq, Hkv, d, N, K_basp)``; the Ulysses layout of the same entry uses
``K = N``.
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    S: int
    Hq: int
    Hkv: int
    d: int
    N: int
    K_basp: int
    dtype: str = "bf16"

    def K(self, layout: str) -> int:
        return self.K_basp if layout == "basp" else self.N

    def tensor_elems(self, H: int) -> int:
        return self.B * self.S * H * self.d


def _family():
    w = [
        # index-valued fp32 correctness shape: B=2, N=4, K=2 (Ulysses K=4)
        Workload("tiny_B2_N4_S64_H4_d16_fp32", 2, 64, 4, 4, 16, 4, 2, "fp32"),
        # Llama-3.2-1B attention: Hq=32, Hkv=8, d=64
        Workload("llama3.2-1b_B2_S8192", 2, 8192, 32, 8, 64, 8, 4),
        # Qwen-1.5-1.8B attention: Hq=Hkv=16, d=128
        Workload("qwen1.5-1.8b_B2_S16384", 2, 16384, 16, 16, 128, 8, 4),
    ]
    # Llama-3.2-3B attention (Hq=24, Hkv=8, d=128), sequence-length sweep
    for S in (1024, 4096, 8192, 16384, 32768):
        w.append(Workload("llama3.2-3b_B2_S%d" % S, 2, S, 24, 8, 128, 8, 4))
    # Llama-3.2-1B micro-batch sweep at S=8192, K = N/B
    for B in (1, 2, 4, 8):
        w.append(Workload("llama3.2-1b_S8192_B%d" % B, B, 8192, 32, 8, 64, 8, 8 // B))
    return w


WORKLOADS = {w.name: w for w in _family()}

# The shape the headline bench line is quoted on: the largest one (Llama-3.2-3B
# heads, B=2, S=32768), the end of the sequence-length sweep.
HEADLINE = "llama3.2-3b_B2_S32768"

# The long-sequence shapes at which the fused kernel should run at >= 80% of the
# HBM copy bandwidth in both directions and both layouts; the bench line
# carries a roofline for each.
TARGETS = ("qwen1.5-1.8b_B2_S16384", "llama3.2-3b_B2_S16384", "llama3.2-3b_B2_S32768")
TARGET_FRACTION = 0.8
