"""Programmatic dependent launch of the short-row kernel.

With ``dependent_launch`` on (the default), the short-row kernel may start
while the kernel before it on the stream is still running; every thread waits
for that kernel's completion before its first global access, and each CTA lets
the next kernel start early in the same way. These tests put calls back to
back on one stream with no synchronisation between them and check that every
call still reads the logits its producer wrote and leaves its own indices in
the output. Every selection is compared with the CPU oracle.
"""
from __future__ import annotations

import numpy as np
import pytest

import workloads
from tests.gpu_util import Runner, assert_matches_oracle

pytestmark = pytest.mark.gpu

ON, OFF = 1, 2

# (workload, rows): whole rows resident (decode_small), whole rows streamed
# (prefill), rows split over clusters of 2 (decode_batch, mtp) and of 6 (long_coop)
CASES = [("decode_small", 8), ("decode_batch", 24), ("mtp", 8), ("long_coop", 4), ("prefill", 320)]


@pytest.fixture(scope="module")
def run():
    return Runner()


def _call(run, x, w, ln, out, opt):
    rc = run.sar.topk_ragged_ex(x, w.row_stride, ln, w.num_rows, w.next_n, w.topk, out, run.sel.workspace,
                                None, opt)
    assert rc == run.sar.TOPK_OK, run.sar.topk_status_string(rc)


def _status_ok(run):
    st = run.sel.status()
    assert st & ~run.sar.TOPK_DEV_LENGTH_CLAMPED == 0, f"device status {st:#x}"


@pytest.mark.parametrize("mode", [0, ON, OFF])
@pytest.mark.parametrize("name,rows", CASES)
def test_back_to_back_calls_into_one_output(run, name, rows, mode):
    # two batches of one shape (the second the negated first, so that their
    # selections differ), selected in turn into the same output: a call whose
    # CTAs start while the one before still runs must write after it, so the
    # output ends with the last batch's selection
    torch = run.torch
    w = workloads.make(name, rows)
    xa = torch.from_numpy(w.logits).to(run.dev)
    xb = torch.from_numpy(-w.logits).to(run.dev)
    ln = torch.from_numpy(w.lengths).to(run.dev)
    out = torch.full((w.num_rows, w.topk), -7, dtype=torch.int32, device=run.dev)
    opt = run.options(dependent_launch=mode)
    for _ in range(8):
        _call(run, xa, w, ln, out, opt)
        _call(run, xb, w, ln, out, opt)
    torch.cuda.synchronize()
    _status_ok(run)
    assert_matches_oracle(-w.logits, w.lengths, out.cpu().numpy(), w.topk, w.next_n,
                          label=f"{name} dependent_launch={mode}")


@pytest.mark.parametrize("mode", [ON, OFF])
@pytest.mark.parametrize("name,rows", [("decode_batch", 24), ("decode_small", 8), ("prefill", 160)])
def test_each_call_reads_what_the_kernel_before_it_wrote(run, name, rows, mode):
    # a copy kernel writes the logits right before each call (no
    # synchronisation): the call must read the new values, and the next copy
    # must not overwrite them before the call is done with them
    torch = run.torch
    w = workloads.make(name, rows)
    rng = np.random.default_rng(7)
    batches = [w.logits * np.float32(s) + np.float32(o)
               for s, o in zip(rng.choice([-1.0, 1.0, 0.5, 2.0], 6), rng.normal(size=6))]
    srcs = [torch.from_numpy(b).to(run.dev) for b in batches]
    x = torch.empty_like(srcs[0])
    ln = torch.from_numpy(w.lengths).to(run.dev)
    outs = [torch.full((w.num_rows, w.topk), -7, dtype=torch.int32, device=run.dev) for _ in batches]
    opt = run.options(dependent_launch=mode)
    torch.cuda.synchronize()
    for src, out in zip(srcs, outs):
        x.copy_(src)
        _call(run, x, w, ln, out, opt)
    torch.cuda.synchronize()
    _status_ok(run)
    for i, (b, out) in enumerate(zip(batches, outs)):
        assert_matches_oracle(b, w.lengths, out.cpu().numpy(), w.topk, w.next_n, label=f"{name} batch {i}")


def test_dependent_launch_value_out_of_range_is_refused(run):
    torch = run.torch
    w = workloads.make("decode_small", 2)
    x = torch.from_numpy(w.logits).to(run.dev)
    ln = torch.from_numpy(w.lengths).to(run.dev)
    out = torch.full((w.num_rows, w.topk), -7, dtype=torch.int32, device=run.dev)
    for bad in (-1, 3):
        rc = run.sar.topk_ragged_ex(x, w.row_stride, ln, w.num_rows, w.next_n, w.topk, out, run.sel.workspace,
                                    None, run.options(dependent_launch=bad))
        assert rc == run.sar.TOPK_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert (out.cpu().numpy() == -7).all()


@pytest.mark.parametrize("name,rows", [("decode_batch", 24), ("mtp", 8), ("prefill", 160)])
def test_selection_then_sort_back_to_back(run, name, rows):
    # selection, then values and order of its rows, for several batches in a
    # row on one stream with no synchronisation: each sort reads the indices
    # its selection wrote, after it has written them all
    import oracle

    torch = run.torch
    sar = run.sar
    w = workloads.make(name, rows)
    R, S = w.logits.shape
    batches = [w.logits, -w.logits, w.logits * np.float32(0.5) + np.float32(1.0)]
    srcs = [torch.from_numpy(b).to(run.dev) for b in batches]
    ln = torch.from_numpy(w.lengths).to(run.dev)
    outs = [torch.full((R, w.topk), -7, dtype=torch.int32, device=run.dev) for _ in batches]
    vals = [torch.zeros((R, w.topk), dtype=torch.float32, device=run.dev) for _ in batches]
    torch.cuda.synchronize()
    for x, out, val in zip(srcs, outs, vals):
        _call(run, x, w, ln, out, run.options())
        assert sar.topk_gather_sort(x, S, 1, S, R, w.topk, out, val, sort=True) == sar.TOPK_OK
    torch.cuda.synchronize()
    _status_ok(run)
    for i, (b, out, val) in enumerate(zip(batches, outs, vals)):
        want, _ = oracle.topk_ragged(b, w.lengths, w.topk, next_n=w.next_n)
        got = out.cpu().numpy()
        assert np.array_equal(got, want), f"{name} batch {i}: rows {np.nonzero((got != want).any(1))[0][:3]}"
        v = val.cpu().numpy()
        ok = got >= 0
        assert np.array_equal(v[ok], b[np.nonzero(ok)[0], got[ok]]) and np.all(np.isneginf(v[~ok]))
