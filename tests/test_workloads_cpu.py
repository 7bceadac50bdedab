"""The seeded input recipe: shapes, length ranges, padding and value mixes.

The bench and the parity tests feed both the CUDA path and the oracle from
``workloads.make``; these checks pin its output to the recipe it documents
(rows, stride, TopK, next_n, how lengths are drawn, what lies beyond them and
what the values look like), so the inputs cannot drift unnoticed.
"""
from __future__ import annotations

import numpy as np
import pytest

import workloads

# (name, rows drawn here, stride, TopK, next_n); prefill is checked on fewer rows
SPECS = [("decode_small", None, 4096, 512, 1), ("decode_batch", None, 32768, 2048, 1),
         ("long_coop", None, 131072, 2048, 1), ("mtp", None, 163840, 1024, 2),
         ("prefill", 96, 65536, 2048, 1)]


def _valid_and_pad(w):
    cols = np.arange(w.row_stride)[None, :]
    inside = cols < np.clip(w.lengths, 0, w.row_stride)[:, None]
    return w.logits[inside], w.logits[~inside]


@pytest.mark.parametrize("name,rows,stride,topk,next_n", SPECS)
def test_shapes_and_padding(name, rows, stride, topk, next_n):
    w = workloads.make(name, rows)
    want_rows = workloads.FULL_ROWS[name] if rows is None else rows
    assert w.logits.shape == (want_rows, stride) and w.logits.dtype == np.float32
    assert w.lengths.shape == (want_rows,) and w.lengths.dtype == np.int32
    assert (w.topk, w.next_n) == (topk, next_n)
    assert w.num_rows % w.next_n == 0
    assert np.all((w.lengths >= 0) & (w.lengths <= stride))
    _, pad = _valid_and_pad(w)
    if name == "mtp":
        assert np.all(np.isneginf(pad))
    else:
        assert np.all(pad == 0.0)
    assert w.valid_bytes() == 4 * int(w.lengths.astype(np.int64).sum())


def test_length_draws():
    assert np.all((workloads.make("decode_small").lengths >= 1) & (workloads.make("decode_small").lengths <= 4096))
    db = workloads.make("decode_batch").lengths
    assert np.all((db >= 8192) & (db <= 32768))
    lc = workloads.make("long_coop").lengths
    assert np.all((lc >= 65536) & (lc <= 131072))
    m = workloads.make("mtp").lengths.reshape(-1, 2)
    assert np.all((m[:, 0] >= 100000) & (m[:, 0] <= 160000))
    assert np.all(m[:, 1] == m[:, 0] + 1)  # row j of a request: L + j
    p = workloads.make("prefill", 96).lengths
    assert np.array_equal(p, 61440 + np.arange(96))


def test_value_mixes():
    # decode_batch: every value on the bfloat16 grid, so exact ties occur
    v, _ = _valid_and_pad(workloads.make("decode_batch"))
    assert np.all((v.view(np.uint32) & np.uint32(0xFFFF)) == 0)
    assert len(np.unique(v)) < v.size // 10
    # long_coop: 10% of entries from N(4, 0.5) on top of N(0, 1)
    v, _ = _valid_and_pad(workloads.make("long_coop"))
    hi = np.mean(v > 2.5)  # N(4, .5) mass above 2.5 is 0.9987; N(0, 1) adds 0.9 * 0.0062
    assert abs(hi - (0.1 * 0.9987 + 0.9 * 0.0062)) < 0.004
    # prefill: 30% exact zeros, a 5% Cauchy tail, the last row all 1.0 (within its length)
    w = workloads.make("prefill", 96)
    body = np.concatenate([w.logits[r, :w.lengths[r]] for r in range(95)])
    assert abs(np.mean(body == 0.0) - 0.30) < 0.005
    assert np.mean(np.abs(body) > 20.0) > 0.05 * 0.02  # Cauchy |x| > 20 has mass 0.0318
    assert np.all(w.logits[95, :w.lengths[95]] == 1.0)
    # decode_small and mtp: plain N(0, 1)
    for name in ("decode_small", "mtp"):
        v, _ = _valid_and_pad(workloads.make(name))
        assert abs(float(v.mean())) < 0.02 and abs(float(v.std()) - 1.0) < 0.02


def test_draws_are_seeded_and_shrinking_keeps_the_recipe():
    a, b = workloads.make("decode_small"), workloads.make("decode_small")
    assert np.array_equal(a.logits, b.logits) and np.array_equal(a.lengths, b.lengths)
    assert a.meta["seed"] == workloads.SEED_BASE + workloads.NAMES.index("decode_small")
    small = workloads.make("long_coop", 4)
    assert small.logits.shape == (4, 131072)
    assert np.all((small.lengths >= 65536) & (small.lengths <= 131072))
    with pytest.raises(ValueError):
        workloads.make("mtp", 3)  # requests contribute two rows each
    with pytest.raises(KeyError):
        workloads.make("no_such_workload")
