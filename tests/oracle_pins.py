"""Pins for the CPU oracle: checks that do not reuse the oracle's own code.

Every pin takes ``mutant`` (0 = the real oracle) and raises AssertionError on a
mismatch. ``test_oracle_pins.py`` runs them on the real oracle;
``test_oracle_mutants.py`` runs them on builds with one planted bug each and
requires that some pin rejects every such build.

What pins the oracle, since the pages print no worked example:
  * brute force on tiny rows: repeated argmax where the first index wins, an
    algorithm with no sorting at all;
  * a library routine: numpy's stable argsort of the negated values;
  * closed forms: constant, increasing and decreasing rows, hand-derived cases;
  * invariants of the selected set on the seeded workloads;
  * torch.topk's values (a third implementation) for the selected multiset.
"""
from __future__ import annotations

import numpy as np

import oracle
import workloads


def run(x, lengths, topk, next_n=1, mutant=0):
    return oracle.topk_ragged(x, lengths, topk, next_n=next_n, mutant=mutant)


def brute_force_row(vals, length, topk):
    """Selection by repeated argmax; a scan in index order keeps the first maximum."""
    length = max(0, min(int(length), len(vals)))
    remaining = list(range(length))
    out = []
    for _ in range(min(length, topk)):
        best = remaining[0]
        for i in remaining[1:]:
            if float(vals[i]) > float(vals[best]):
                best = i
        out.append(best)
        remaining.remove(best)
    return out + [-1] * (topk - len(out))


def pin_brute_force(mutant=0, trials=400, seed=7):
    rng = np.random.default_rng(seed)
    for _ in range(trials):
        stride = int(rng.integers(1, 13))
        rows = int(rng.integers(1, 4))
        x, lengths = workloads.tiny_rows(rng, rows, stride)
        topk = int(rng.integers(1, 9))
        got, _ = run(x, lengths, topk, mutant=mutant)
        for r in range(rows):
            want = brute_force_row(x[r], lengths[r], topk)
            assert got[r].tolist() == want, (x[r].tolist(), int(lengths[r]), topk, got[r].tolist(), want)


def pin_numpy_argsort(mutant=0, seed=11):
    rng = np.random.default_rng(seed)
    for topk in (1, 7, 512, 1024, 2048):
        for stride in (1, 5, 600, 3000):
            rows = 3
            x = rng.standard_normal((rows, stride)).astype(np.float32)
            # coarse grid so that exact ties are common
            x = np.round(x * 8) / 8
            lengths = rng.integers(0, stride, size=rows, endpoint=True).astype(np.int32)
            got, _ = run(x.astype(np.float32), lengths, topk, mutant=mutant)
            for r in range(rows):
                n = int(lengths[r])
                order = np.argsort(-x[r, :n], kind="stable")[:topk]
                want = np.full(topk, -1, dtype=np.int64)
                want[: len(order)] = order
                assert np.array_equal(got[r], want), (topk, stride, r)


def pin_closed_forms(mutant=0):
    K = 512
    # constant row: the first K indices
    x = np.full((1, 3000), 0.25, dtype=np.float32)
    got, _ = run(x, np.array([3000], np.int32), K, mutant=mutant)
    assert got[0].tolist() == list(range(K))
    # strictly increasing row: the last K indices, largest first
    x = np.arange(3000, dtype=np.float32)[None, :]
    got, _ = run(x, np.array([2500], np.int32), K, mutant=mutant)
    assert got[0].tolist() == list(range(2499, 2499 - K, -1))
    # strictly decreasing row: the first K indices
    x = -np.arange(3000, dtype=np.float32)[None, :]
    got, _ = run(x, np.array([2999], np.int32), K, mutant=mutant)
    assert got[0].tolist() == list(range(K))
    # rows no longer than K: every valid index, by value, then -1
    x = np.array([[2.0, -1.0, 5.0, 5.0, 9.0]], dtype=np.float32)
    got, _ = run(x, np.array([4], np.int32), 8, mutant=mutant)
    assert got[0].tolist() == [2, 3, 0, 1, -1, -1, -1, -1]
    # empty row
    got, _ = run(x, np.array([0], np.int32), 3, mutant=mutant)
    assert got[0].tolist() == [-1, -1, -1]


# Hand-derived cases: (row values, length, topk, expected), each worked out from
# the selection rule (larger value first, smaller index on equal values, -1
# padding after min(length, topk) indices).
HAND_CASES = [
    # 3.0@1 and 3.0@3 tie: index 1 first; then 2.0@2
    ([1.0, 3.0, 2.0, 3.0, -1.0], 5, 3, [1, 3, 2]),
    # -0.0 equals +0.0: after 5.0@3 the zeros come in index order 0, 1, 2
    ([-0.0, 0.0, -0.0, 5.0], 4, 4, [3, 0, 1, 2]),
    # two valid values, four slots
    ([2.0, 1.0], 2, 4, [0, 1, -1, -1]),
    # +inf first, then the smallest subnormal, which is above 0.0
    ([np.inf, -np.inf, 1e-45, 0.0], 4, 2, [0, 2]),
    # the 9.0 at index 3 lies beyond the length and is never chosen
    ([7.0, 7.0, 7.0, 9.0], 3, 2, [0, 1]),
    # -5.0 beats -inf; the two -inf tie and go in index order
    ([-np.inf, -np.inf, -5.0, -np.inf], 4, 3, [2, 0, 1]),
    # subnormals are ordered exactly: 2x the smallest beats 1x
    ([1e-45, 3e-45, -1e-45, 0.0], 4, 2, [1, 0]),
]


def pin_hand_cases(mutant=0):
    for vals, length, topk, want in HAND_CASES:
        x = np.array([vals], dtype=np.float32)
        got, st = run(x, np.array([length], np.int32), topk, mutant=mutant)
        assert got[0].tolist() == want, (vals, length, topk, got[0].tolist(), want)
        assert st == 0


def pin_length_clamp(mutant=0):
    x = np.array([[1.0, 2.0, 3.0]], dtype=np.float32)
    got, st = run(x, np.array([10], np.int32), 2, mutant=mutant)
    assert got[0].tolist() == [2, 1] and st & oracle.STATUS_LENGTH_CLAMPED
    got, st = run(x, np.array([-5], np.int32), 2, mutant=mutant)
    assert got[0].tolist() == [-1, -1] and st & oracle.STATUS_LENGTH_CLAMPED


def pin_mtp_rows(mutant=0):
    # one request, next_n = 2: row j has length L + j, so row 1 sees index 4
    x = np.array([[0.0, 1.0, 2.0, 3.0, 100.0, 0.0],
                  [0.0, 1.0, 2.0, 3.0, 100.0, 0.0]], dtype=np.float32)
    got, _ = run(x, np.array([4, 5], np.int32), 2, next_n=2, mutant=mutant)
    assert got.tolist() == [[3, 2], [4, 3]], got.tolist()


def check_invariants(x_row, length, sel, topk):
    """The selected set is the top-K under (value desc, index asc); raises on violation."""
    n = max(0, min(int(length), x_row.shape[0]))
    take = min(n, topk)
    assert np.all(sel[take:] == -1), "padding must be -1"
    s = sel[:take].astype(np.int64)
    assert np.all((s >= 0) & (s < n)), "indices must lie in [0, len)"
    assert len(np.unique(s)) == take, "indices must be distinct"
    if take == 0 or take == n:
        return
    v = x_row[:n]
    mask = np.zeros(n, dtype=bool)
    mask[s] = True
    vmin = v[mask].min()
    vmax_un = v[~mask].max()
    assert vmin >= vmax_un, "every selected value must be >= every unselected value"
    if vmin == vmax_un:  # ties at the threshold: selected indices come first
        tie_sel = np.nonzero(mask & (v == vmin))[0]
        tie_un = np.nonzero(~mask & (v == vmin))[0]
        assert tie_sel.max() < tie_un.min(), "ties must go to the smaller indices"


def pin_workload_invariants(mutant=0):
    import torch

    for name, rows in (("decode_small", 8), ("decode_batch", 6), ("long_coop", 2), ("mtp", 4),
                       ("prefill", 3)):
        w = workloads.make(name, rows)
        got, _ = run(w.logits, w.lengths, w.topk, next_n=w.next_n, mutant=mutant)
        for r in range(w.num_rows):
            check_invariants(w.logits[r], w.lengths[r], got[r], w.topk)
            n = int(w.lengths[r])
            take = min(n, w.topk)
            if take:
                tv = torch.topk(torch.from_numpy(w.logits[r, :n].copy()), take).values.numpy()
                sv = np.sort(w.logits[r][got[r][:take]])[::-1]
                assert np.array_equal(sv, tv), "selected values must be the top-K multiset"


ALL_PINS = [pin_brute_force, pin_numpy_argsort, pin_closed_forms, pin_hand_cases,
            pin_length_clamp, pin_mtp_rows, pin_workload_invariants]

MUTANTS = {
    1: "ties go to the larger index",
    2: "pads with 0 instead of -1",
    3: "drops the last valid element",
    4: "orders -0.0 below +0.0",
    6: "selects the smallest values",
    7: "one index short at the topk boundary",
    10: "addresses rows by length instead of stride",
    11: "one length per request instead of per row",
}
