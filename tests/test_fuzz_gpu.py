"""Seeded random sweep over launch shapes, merges, TopK and row mixes, against the oracle.

Each case draws a batch (rows, stride, lengths, next_n), a TopK and a plan
(CTA shape, merge kind, forced split size) from a fixed seed, runs it through
topk_ragged_ex and compares every row with the oracle element by element
(after ordering by the tie rule), then checks the workspace is back to zero.
Rows mix value distributions that stress different paths: ties on a small
alphabet, all-equal rows (buffer overflow and re-stream), increasing rows
(the seed undershoots), +-0 and +-inf, bf16-rounded normals.
"""
from __future__ import annotations

import os

import numpy as np
import pytest

from tests.gpu_util import Runner, assert_matches_oracle

pytestmark = pytest.mark.gpu

# TOPK_FUZZ_CASES=N runs N seeds of every generator below instead of their defaults
FUZZ_CASES = int(os.environ.get("TOPK_FUZZ_CASES", "0"))
CASES = FUZZ_CASES or 80
MAX_ELEMENTS = 3_000_000  # keeps the oracle to well under a second per case


@pytest.fixture(scope="module")
def rn():
    return Runner()


def _row(rng: np.random.Generator, n: int) -> np.ndarray:
    kind = rng.integers(0, 9)
    if kind == 0:
        return rng.standard_normal(n).astype(np.float32)
    if kind == 1:  # bf16 grid: many equal values
        x = rng.standard_normal(n).astype(np.float32)
        return (x.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)
    if kind == 2:  # small alphabet with signed zeros and infinities
        a = np.array([-np.inf, -1.0, -0.0, 0.0, 0.5, 1.0, 2.0, np.inf], np.float32)
        return rng.choice(a, size=n).astype(np.float32)
    if kind == 3:
        return np.full(n, np.float32(rng.standard_normal()), np.float32)
    if kind == 4:
        return np.arange(n, dtype=np.float32) * np.float32(rng.choice([1.0, -1.0]))
    if kind == 5:  # a few large values over a flat floor
        x = np.full(n, -3.0, np.float32)
        k = int(rng.integers(1, max(2, n // 8)))
        x[rng.choice(n, size=min(k, n), replace=False)] = rng.standard_normal(min(k, n)).astype(np.float32) + 5
        return x
    if kind == 6:  # heavy tails
        return rng.standard_cauchy(n).astype(np.float32)
    if kind == 8:  # a dense cluster: many elements share the K-th key's top bits
        x = rng.standard_normal(n).astype(np.float32)
        m = rng.random(n) < rng.uniform(0.02, 0.3)
        x[m] = (4.0 + rng.choice([0.02, 0.1, 0.3]) * rng.standard_normal(int(m.sum()))).astype(np.float32)
        return x
    return (rng.standard_normal(n) * 0.01).astype(np.float32)


def _case(seed: int):
    rng = np.random.default_rng(1_000_003 * seed + 17)
    shape = int(rng.choice([0, 0, 1, 2, 3]))
    kmax = 4096 if shape in (0, 1) else 2048
    topk = int(rng.choice([int(rng.integers(1, 65)), 512, 1024, 2048, int(rng.integers(1, kmax + 1))]))
    topk = min(topk, kmax)
    next_n = int(rng.choice([1, 1, 2, 3]))
    stride = int(rng.choice([int(rng.integers(1, 5000)), int(rng.integers(5000, 40000)),
                             int(rng.integers(40000, 140000))]))
    max_rows = max(1, min(300, MAX_ELEMENTS // stride))
    num_rows = int(rng.integers(1, max_rows + 1))
    num_rows = max(next_n, num_rows - num_rows % next_n)
    force, merge = 0, 0
    if shape in (0, 1) and rng.random() < 0.5:
        force = int(rng.choice([1, 2, 3, 4, 6, 8]))
        merge = int(rng.choice([0, 1, 2]))
    x = np.stack([_row(rng, stride) for _ in range(num_rows)])
    lengths = rng.integers(0, stride + 1, size=num_rows)
    full = rng.random(num_rows) < 0.3
    lengths[full] = stride
    short = rng.random(num_rows) < 0.1
    lengths[short] = rng.integers(0, min(topk, stride) + 1, size=int(short.sum()))
    if next_n > 1:  # one length per request: row j of a request sees len + j
        base = lengths.reshape(-1, next_n)[:, 0]
        lengths = np.minimum(base[:, None] + np.arange(next_n)[None, :], stride).reshape(-1)
    return x, lengths.astype(np.int32), topk, next_n, dict(shape=shape, force_ctas_per_group=force, merge=merge)


@pytest.mark.parametrize("seed", range(CASES))
def test_random_case_matches_oracle(rn, seed):
    x, lengths, topk, next_n, opts = _case(seed)
    got = rn.run(x, lengths, topk, next_n=next_n, options=rn.options(**opts))
    assert_matches_oracle(x, lengths, got, topk, next_n=next_n,
                          label=f"seed {seed}: {x.shape[0]} rows x {x.shape[1]}, K {topk}, next_n {next_n}, {opts}")
    assert rn.workspace_clean()


SHORT_CASES = FUZZ_CASES or 40


def _short_case(seed: int):
    """Batches for the short-row kernel: rows resident in its ring (up to 32768 elements) and
    rows streamed through it (up to 140000), one CTA per row or several rows per CTA, every value
    mix, TopK up to 4096."""
    rng = np.random.default_rng(2_000_029 * seed + 5)
    topk = int(rng.choice([int(rng.integers(1, 65)), 512, 1024, 2048, int(rng.integers(1, 4097))]))
    stride = int(rng.choice([int(rng.integers(1, 5000)), int(rng.integers(5000, 32769)), 32768,
                             int(rng.integers(32769, 140000))]))
    num_rows = int(rng.integers(1, min(200, MAX_ELEMENTS // stride) + 1))
    x = np.stack([_row(rng, stride) for _ in range(num_rows)])
    lengths = rng.integers(0, stride + 1, size=num_rows)
    lengths[rng.random(num_rows) < 0.3] = stride
    max_ctas = int(rng.choice([0, 0, 1, 3, 17]))
    return x, lengths.astype(np.int32), topk, dict(shape=int(rng.choice([4, 5])), max_ctas=max_ctas,
                                                   force_ctas_per_group=1)


@pytest.mark.parametrize("seed", range(SHORT_CASES))
def test_random_short_rows_match_oracle(rn, seed):
    x, lengths, topk, opts = _short_case(seed)
    got = rn.run(x, lengths, topk, options=rn.options(**opts))
    assert_matches_oracle(x, lengths, got, topk,
                          label=f"short seed {seed}: {x.shape[0]} rows x {x.shape[1]}, K {topk}, {opts}")


CLUSTER_CASES = FUZZ_CASES or 40


def _cluster_case(seed: int):
    """Rows split over a thread-block cluster of the short-row kernel (2 to 8 CTAs, one row per
    cluster): lengths from below TopK to past the ring of every CTA, every value mix, TopK up to
    4096, row starts off the 16-byte grid."""
    rng = np.random.default_rng(3_000_017 * seed + 11)
    G = int(rng.integers(2, 9))
    topk = int(rng.choice([int(rng.integers(1, 65)), 512, 1024, 2048, int(rng.integers(1, 4097))]))
    stride = int(rng.choice([int(rng.integers(1, 8000)), int(rng.integers(8000, 70000)),
                             int(rng.integers(70000, 300000))]))
    num_rows = int(rng.integers(1, min(40, MAX_ELEMENTS // stride) + 1))
    x = np.stack([_row(rng, stride) for _ in range(num_rows)])
    lengths = rng.integers(0, stride + 1, size=num_rows)
    lengths[rng.random(num_rows) < 0.3] = stride
    return x, lengths.astype(np.int32), topk, int(rng.integers(0, 4)), dict(shape=int(rng.choice([4, 5])),
                                                                           force_ctas_per_group=G)


@pytest.mark.parametrize("seed", range(CLUSTER_CASES))
def test_random_cluster_split_rows_match_oracle(rn, seed):
    x, lengths, topk, shift, opts = _cluster_case(seed)
    got = rn.run(x, lengths, topk, options=rn.options(**opts), pad_front=shift)
    assert_matches_oracle(x, lengths, got, topk,
                          label=f"cluster seed {seed}: {x.shape[0]} rows x {x.shape[1]}, K {topk}, shift {shift}, "
                                f"{opts}")
