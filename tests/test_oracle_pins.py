"""The CPU oracle against brute force, numpy, closed forms and invariants."""
import numpy as np
import pytest

import oracle
import workloads
from tests import oracle_pins as P


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(mutant=0)


def test_threads_do_not_change_the_result():
    w = workloads.make("prefill", 24)
    a, _ = oracle.topk_ragged(w.logits, w.lengths, w.topk, nthreads=1)
    b, _ = oracle.topk_ragged(w.logits, w.lengths, w.topk, nthreads=7)
    assert np.array_equal(a, b)


def test_rejects_bad_arguments():
    x = np.zeros((3, 4), np.float32)
    with pytest.raises(ValueError):
        oracle.topk_ragged(x, np.array([1, 2, 3], np.int32), 2, next_n=2)


def test_workload_recipes():
    w = workloads.make("decode_batch", 8)
    # values on the bf16 grid: the low 16 bits are zero
    assert np.all((w.logits.view(np.uint32) & 0xFFFF) == 0)
    assert w.lengths.min() >= 8192 and w.lengths.max() <= 32768
    m = workloads.make("mtp", 6)
    assert np.all(m.lengths[1::2] == m.lengths[0::2] + 1)
    assert np.isneginf(m.logits[0, m.lengths[0]:]).all()
    p = workloads.make("prefill", 5)
    assert p.lengths.tolist() == [61440 + i for i in range(5)]
    assert np.all(p.logits[4, : p.lengths[4]] == 1.0)
    frac0 = np.mean(p.logits[0, : p.lengths[0]] == 0.0)
    assert 0.28 < frac0 < 0.32
