"""Workspace hygiene: no per-call memset, graph replay, bounded waits (GPU only)."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import workloads
from tests.gpu_util import Runner, assert_matches_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rn():
    return Runner()


def test_back_to_back_calls_share_one_workspace(rn):
    """Alternating shapes and both paths, with no clearing between calls."""
    cases = []
    for name, rows in (("long_coop", 3), ("decode_batch", 8), ("mtp", 4), ("decode_small", 8)):
        w = workloads.make(name, rows)
        want, _ = oracle.topk_ragged(w.logits, w.lengths, w.topk, next_n=w.next_n)
        cases.append((w, want))
    rn.sel.reset()
    for i in range(120):
        w, want = cases[i % len(cases)]
        G, merge = ((0, 0), (1, 0), (2, 1), (7, 2), (2, 2), (7, 1))[(i // len(cases)) % 6]
        got = rn.run(w.logits, w.lengths, w.topk, w.next_n,
                     options=rn.options(force_ctas_per_group=G, merge=merge))
        if i % 7 == 0 or i >= 112:
            assert_matches_oracle(w.logits, w.lengths, got, w.topk, w.next_n, want=want,
                                  label=f"call {i} {w.name} G={G}")
    assert rn.workspace_clean()
    assert rn.sel.status() == 0


@pytest.mark.parametrize("merge", [1, 2])
def test_graph_replay_with_changing_inputs(rn, merge):
    torch = rn.torch
    sar = rn.sar
    rows, S, K = 12, 131072, 2048
    xs = torch.zeros((rows, S), dtype=torch.float32, device=rn.dev)
    ls = torch.zeros(rows, dtype=torch.int32, device=rn.dev)
    out = torch.zeros((rows, K), dtype=torch.int32, device=rn.dev)
    opts = rn.options(force_ctas_per_group=6, merge=merge)
    # first call outside capture (device properties are cached on it)
    assert sar.topk_ragged_ex(xs, S, ls, rows, 1, K, out, rn.sel.workspace, None, opts) == 0
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        rc = sar.topk_ragged_ex(xs, S, ls, rows, 1, K, out, rn.sel.workspace, None, opts)
    assert rc == 0
    rng = np.random.default_rng(4)
    for it in range(6):
        x = rng.standard_normal((rows, S)).astype(np.float32)
        if it % 2:
            x = np.round(x * 16) / 16
        lens = rng.integers(0, S, rows, endpoint=True).astype(np.int32)
        xs.copy_(torch.from_numpy(x))
        ls.copy_(torch.from_numpy(lens))
        g.replay()
        torch.cuda.synchronize()
        assert_matches_oracle(x, lens, out.cpu().numpy(), K, label=f"replay {it}")
        assert rn.workspace_clean()


def test_timed_out_group_wait_reports_and_recovers(rn):
    """A CTA that never arrives makes its partners' bounded waits run out."""
    w = workloads.make("long_coop", 4)
    rn.sel.reset()
    opts = rn.options(force_ctas_per_group=2, merge=1, inject_skip_arrival=1, barrier_timeout_us=20000)
    rn.run(w.logits, w.lengths, w.topk, options=opts, check_status=False)
    st = rn.sel.status()
    assert st & rn.sar.TOPK_DEV_BARRIER_TIMEOUT, f"status {st:#x}"
    # the context is still usable; re-initialising the workspace restores service
    rn.sel.reset()
    got = rn.run(w.logits, w.lengths, w.topk, options=rn.options(force_ctas_per_group=2, merge=1))
    assert_matches_oracle(w.logits, w.lengths, got, w.topk, label="after recovery")
    assert rn.workspace_clean()


def test_dirty_workspace_is_refused_not_merged(rn):
    """After a time-out the group words are stale; a later split launch must not merge through them.

    Without topk_workspace_init, the next call that splits rows writes rows of -1 and sets
    TOPK_DEV_WORKSPACE_DIRTY (wrong indices with a clean status would be the failure); whole-row
    calls never read the group words and stay exact.
    """
    sar = rn.sar
    w = workloads.make("long_coop", 4)
    rn.sel.reset()
    opts = rn.options(force_ctas_per_group=2, merge=1, inject_skip_arrival=1, barrier_timeout_us=20000)
    rn.run(w.logits, w.lengths, w.topk, options=opts, check_status=False)
    assert rn.sel.status() & sar.TOPK_DEV_BARRIER_TIMEOUT
    for G, merge in ((2, 1), (4, 2)):
        got = rn.run(w.logits, w.lengths, w.topk, options=rn.options(force_ctas_per_group=G, merge=merge),
                     check_status=False)
        assert rn.sel.status() & sar.TOPK_DEV_WORKSPACE_DIRTY, f"G={G} merge={merge}"
        assert (got == -1).all(), f"G={G} merge={merge}: a refused launch writes rows of -1"
    got = rn.run(w.logits, w.lengths, w.topk, options=rn.options(force_ctas_per_group=1), check_status=False)
    assert_matches_oracle(w.logits, w.lengths, got, w.topk, label="whole rows on a dirty workspace")
    rn.sel.reset()
    got = rn.run(w.logits, w.lengths, w.topk, options=rn.options(force_ctas_per_group=2, merge=1))
    assert_matches_oracle(w.logits, w.lengths, got, w.topk, label="after re-initialisation")
    assert rn.workspace_clean()


@pytest.mark.parametrize("G", [2, 4])
def test_timed_out_cluster_sync_reports_and_every_cta_leaves(rn, G):
    """A cluster member that withholds its merge arrivals: every member's bounded wait runs out,
    the launch ends (all CTAs meet at the cluster's exit barrier), and the context stays usable."""
    sar = rn.sar
    w = workloads.make("long_coop", 3)
    rn.sel.reset()
    opts = rn.options(force_ctas_per_group=G, merge=2, inject_skip_arrival=2, barrier_timeout_us=20000)
    rn.run(w.logits, w.lengths, w.topk, options=opts, check_status=False)
    st = rn.sel.status()
    assert st & sar.TOPK_DEV_BARRIER_TIMEOUT, f"status {st:#x}"
    assert not st & sar.TOPK_DEV_STAGE_TIMEOUT, f"status {st:#x}: the members' copies all landed"
    rn.sel.reset()
    got = rn.run(w.logits, w.lengths, w.topk, options=rn.options(force_ctas_per_group=G, merge=2))
    assert_matches_oracle(w.logits, w.lengths, got, w.topk, label=f"cluster G={G} after recovery")
    assert rn.workspace_clean()


@pytest.mark.parametrize("shape,G,name,rows", [(5, 2, "decode_batch", 8), (5, 6, "long_coop", 4), (4, 3, "mtp", 4),
                                               (5, 8, "long_coop", 3)])
def test_short_row_cta_that_gives_up_leaves_cleanly(rn, shape, G, name, rows):
    """A CTA of a row split over a short-row cluster that gives up (host-chosen: it treats its
    first copy as late, after the copy has landed) flags TOPK_DEV_STAGE_TIMEOUT; every CTA of its
    cluster leaves through the same barriers, row 0 is left unwritten and every other row is
    selected exactly."""
    sar = rn.sar
    w = workloads.make(name, rows)
    assert w.lengths[0] > w.topk  # row 0 reaches the copy wait
    rn.sel.reset()
    opts = rn.options(shape=shape, force_ctas_per_group=G, inject_skip_arrival=3)
    got = rn.run(w.logits, w.lengths, w.topk, w.next_n, options=opts, check_status=False)
    st = rn.sel.status()
    assert st & sar.TOPK_DEV_STAGE_TIMEOUT, f"status {st:#x}"
    assert not st & sar.TOPK_DEV_BARRIER_TIMEOUT, f"status {st:#x}"
    assert (got[0] == -7).all(), "the row of the CTA that gave up is left as it was"
    assert_matches_oracle(w.logits[1:], w.lengths[1:], got[1:], w.topk, label=f"{name} other rows")
    rn.sel.reset()
    got = rn.run(w.logits, w.lengths, w.topk, w.next_n, options=rn.options(shape=shape, force_ctas_per_group=G))
    assert_matches_oracle(w.logits, w.lengths, got, w.topk, w.next_n, label=f"{name} after the injected give-up")
