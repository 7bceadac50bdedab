"""Seeded synthetic inputs for the ragged per-row top-K.

This module only draws random inputs; it holds none of the selection
arithmetic. Tests, the smoke check and ``bench.py`` use it to feed both the
CUDA path and the CPU oracle the same rows.

Five workloads, each with its shapes, value distributions and length mix:

=============  ======  ========================  ========  ====  ==============================  ======
name           rows    lengths                   stride    TopK  values                          next_n
=============  ======  ========================  ========  ====  ==============================  ======
decode_small   8       uniform int in [1, 4096]   4096     512   N(0,1)                          1
decode_batch   64      uniform int [8192, 32768]  32768    2048  N(0,1) rounded to bf16 (ties)   1
long_coop      16      uniform [65536, 131072]    131072   2048  90% N(0,1) + 10% N(4, sd 0.5)   1
mtp            32x2    L ~ U[100000,160000], L+j  163840   1024  N(0,1), -inf beyond the length  2
prefill        4096    61440 + i                  65536    2048  30% 0.0, 5% Cauchy, 65% N(0,1)  1
=============  ======  ========================  ========  ====  ==============================  ======

``prefill`` also sets its last row to all 1.0 (the "one row that is all
equal"). Padding beyond each length is 0.0 except in ``mtp`` (-inf).
Every draw comes from ``numpy.random.default_rng(20260 + index)`` (PCG64),
where ``index`` is the workload's position in the table (0..4). Integer
"uniform in [a, b]" includes both ends. Smaller variants (fewer rows or
requests, same per-row recipe) serve the parity tests.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

SEED_BASE = 20260


@dataclass
class Workload:
    name: str
    logits: np.ndarray          # float32 [num_rows, row_stride]
    lengths: np.ndarray         # int32 [num_rows]
    topk: int
    next_n: int
    meta: dict = field(default_factory=dict)

    @property
    def num_rows(self) -> int:
        return int(self.logits.shape[0])

    @property
    def row_stride(self) -> int:
        return int(self.logits.shape[1])

    def valid_bytes(self) -> int:
        """Bytes of valid logits (sum of 4 * clamp(len, 0, stride))."""
        ln = np.clip(self.lengths.astype(np.int64), 0, self.row_stride)
        return int(4 * ln.sum())


NAMES = ("decode_small", "decode_batch", "long_coop", "mtp", "prefill")

FULL_ROWS = {"decode_small": 8, "decode_batch": 64, "long_coop": 16, "mtp": 64, "prefill": 4096}


def _bf16_round(x: np.ndarray) -> np.ndarray:
    """Rounds float32 values to the nearest bfloat16 (ties to even), kept as float32."""
    u = x.view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) & np.uint32(0xFFFF0000)).view(np.float32)


def make(name: str, num_rows: int | None = None) -> Workload:
    """Builds workload ``name``; ``num_rows`` shrinks it (rows, or 2 x requests for mtp)."""
    if name not in NAMES:
        raise KeyError(name)
    index = NAMES.index(name)
    rng = np.random.default_rng(SEED_BASE + index)
    n = FULL_ROWS[name] if num_rows is None else int(num_rows)
    if name == "decode_small":
        S, K, nn = 4096, 512, 1
        lengths = rng.integers(1, 4096, size=n, endpoint=True)
        x = rng.standard_normal((n, S), dtype=np.float32)
        pad = 0.0
    elif name == "decode_batch":
        S, K, nn = 32768, 2048, 1
        lengths = rng.integers(8192, 32768, size=n, endpoint=True)
        x = _bf16_round(rng.standard_normal((n, S), dtype=np.float32))
        pad = 0.0
    elif name == "long_coop":
        S, K, nn = 131072, 2048, 1
        lengths = rng.integers(65536, 131072, size=n, endpoint=True)
        x = rng.standard_normal((n, S), dtype=np.float32)
        hi = rng.random((n, S), dtype=np.float32) < np.float32(0.10)
        x[hi] = (np.float32(4.0) + np.float32(0.5) * x[hi]).astype(np.float32)
        pad = 0.0
    elif name == "mtp":
        S, K, nn = 163840, 1024, 2
        if n % nn:
            raise ValueError("mtp needs an even number of rows")
        base = rng.integers(100000, 160000, size=n // nn, endpoint=True)
        lengths = (base[:, None] + np.arange(nn)[None, :]).reshape(-1)
        x = rng.standard_normal((n, S), dtype=np.float32)
        pad = -np.inf
    else:  # prefill
        S, K, nn = 65536, 2048, 1
        lengths = 61440 + np.arange(n)
        x = rng.standard_normal((n, S), dtype=np.float32)
        u = rng.random((n, S), dtype=np.float32)
        x[u < np.float32(0.30)] = 0.0
        cau = (u >= np.float32(0.30)) & (u < np.float32(0.35))
        x[cau] = rng.standard_cauchy(int(cau.sum())).astype(np.float32)
        x[n - 1, :] = 1.0
        pad = 0.0
    lengths = np.minimum(lengths, S).astype(np.int32)
    cols = np.arange(S)[None, :]
    x[cols >= lengths[:, None]] = pad
    return Workload(name, np.ascontiguousarray(x), lengths, K, nn,
                    {"index": index, "seed": SEED_BASE + index, "full_rows": FULL_ROWS[name]})


def tiny_rows(rng: np.random.Generator, num_rows: int, row_stride: int, alphabet=None,
              with_specials: bool = True) -> tuple[np.ndarray, np.ndarray]:
    """Small rows over a small value alphabet so that ties, +-0 and +-inf occur."""
    if alphabet is None:
        alphabet = np.array([-2.0, -1.0, -0.0, 0.0, 0.5, 1.0, 1.0, 3.0], dtype=np.float32)
        if with_specials:
            alphabet = np.concatenate([alphabet, np.array([np.inf, -np.inf, 1e-45, -1e-45],
                                                          dtype=np.float32)])
    x = rng.choice(alphabet, size=(num_rows, row_stride)).astype(np.float32)
    lengths = rng.integers(0, row_stride, size=num_rows, endpoint=True).astype(np.int32)
    return x, lengths
