"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module draws numbers only: it holds none of the re-layout's arithmetic
(no shard, rank or head index math), so the CUDA path and the oracle can both
take their inputs from it without sharing any of the method.

Workload shapes (the attention activations of Llama-3.2-1B / -3B and
Qwen-1.5-1.8B are used as shape labels only: no weights, no data):

* values ~N(0, 1), drawn in fp32 from a CPU ``torch.Generator`` seeded with
  ``seed``, then rounded to the target dtype;
* index-valued inputs: element i of a flat buffer holds ``offset + i``
  (exact in fp32 while below 2**24).
"""
from __future__ import annotations

import numpy as np
import torch

DTYPES = {
    "bf16": torch.bfloat16,
    "fp16": torch.float16,
    "fp32": torch.float32,
    "fp8": torch.float8_e4m3fn,
}

# numpy view types for comparing raw bits
BITS = {
    torch.bfloat16: torch.int16,
    torch.float16: torch.int16,
    torch.float32: torch.int32,
    torch.float8_e4m3fn: torch.int8,
}


def normal(n: int, seed: int, dtype: str = "bf16") -> torch.Tensor:
    """``n`` values ~N(0,1) on the CPU, rounded to ``dtype``."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    x = torch.randn(int(n), generator=g, dtype=torch.float32)
    return x.to(DTYPES[dtype])


def random_bits(n: int, seed: int, dtype: str = "bf16") -> torch.Tensor:
    """``n`` elements whose bit patterns are uniform (NaN payloads, -0,
    subnormals and infinities included), on the CPU."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    t = DTYPES[dtype]
    bt = BITS[t]
    info = torch.iinfo(bt)
    x = torch.randint(info.min, info.max + 1, (int(n),), generator=g,
                      dtype=torch.int64).to(bt)
    return x.view(t)


def index_valued(n: int, offset: int = 0) -> torch.Tensor:
    """fp32 buffer whose element i holds ``offset + i``."""
    if offset + n > (1 << 24):
        raise ValueError("index values above 2**24 are not exact in fp32")
    return torch.arange(offset, offset + int(n), dtype=torch.float32)


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw bits of a CPU tensor as a numpy integer array."""
    return t.contiguous().view(BITS[t.dtype]).numpy()


def normal_device(n: int, seed: int, dtype: str, device) -> torch.Tensor:
    """Like :func:`normal`, drawn by the device's own generator (the bench's
    full-size buffers; the values differ from the CPU draw of the same seed)."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.randn(int(n), generator=g, dtype=torch.float32, device=device)
    return x.to(DTYPES[dtype])


def random_bits_device(n: int, seed: int, dtype: str, device) -> torch.Tensor:
    """Like :func:`random_bits`, drawn by the device's own generator (for
    buffers too large to draw on the CPU in a test's time)."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    t = DTYPES[dtype]
    bt = BITS[t]
    info = torch.iinfo(bt)
    x = torch.randint(info.min, info.max + 1, (int(n),), generator=g,
                      dtype=bt, device=device)
    return x.view(t)
