"""topk_ragged_static (no workspace, no allocation) against the oracle.

Callers that cannot allocate device memory use topk_ragged_static, whose
scratch is a fixed array inside the library. This file runs last so that a
failure here never hides another test; it also passes on its own, in a fresh
process (the first call on the device then sets the array up).
"""
import numpy as np
import pytest

import oracle
import workloads
from tests.gpu_util import Runner, assert_matches_oracle

pytestmark = pytest.mark.gpu


def _run_static(rn, x, lengths, topk, next_n=1):
    torch = rn.torch
    rows, stride = x.shape
    xd = torch.from_numpy(np.ascontiguousarray(x)).to(rn.dev)
    ln = torch.from_numpy(np.ascontiguousarray(lengths, dtype=np.int32)).to(rn.dev)
    out = torch.full((rows, topk), -7, dtype=torch.int32, device=rn.dev)
    rc = rn.sar.topk_ragged_static(xd, stride, ln, rows, next_n, topk, out)
    assert rc == rn.sar.TOPK_OK, rn.sar.topk_status_string(rc)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _plan(rn, rows, stride, next_n, topk):
    props = rn.sar.topk_query_device(rn.dev.index)
    rc, pl = rn.sar.topk_make_plan(props, rows, stride, next_n, topk)
    assert rc == 0
    return pl


def test_static_matches_the_oracle_on_two_calls_in_a_row():
    rn = Runner()
    # rows split over clusters (long_coop, mtp), whole rows (decode_batch), and rows
    # split eight ways whose all-equal values overflow the cluster leader, so the
    # members merge through the row-group areas of the fixed array
    S = 1 << 20  # rows this long are split across CTAs
    tied = np.ones((4, S), np.float32)
    tied[1, ::3] = 2.0
    tied_lens = np.array([S, S, 700000, 300001], np.int32)
    pl = _plan(rn, 4, S, 1, 2048)
    assert pl.ctas_per_group == 8 and pl.cluster, "the tied case is planned as clusters of eight"
    cases = [(w.name, w.logits, w.lengths, w.topk, w.next_n)
             for w in (workloads.make("long_coop", 3), workloads.make("decode_batch", 10), workloads.make("mtp", 4))]
    cases.append(("tied", tied, tied_lens, 2048, 1))
    for call in range(2):
        for name, x, lens, topk, next_n in cases:
            want, _ = oracle.topk_ragged(x, lens, topk, next_n=next_n)
            got = _run_static(rn, x, lens, topk, next_n)
            assert_matches_oracle(x, lens, got, topk, next_n, want=want, label=f"static call {call} {name}")
    # a changed batch through the same scratch
    w = workloads.make("long_coop", 3)
    rng = np.random.default_rng(77)
    x = np.round(rng.standard_normal(w.logits.shape) * 8).astype(np.float32) / 8
    assert_matches_oracle(x, w.lengths, _run_static(rn, x, w.lengths, w.topk), w.topk, label="static changed batch")
