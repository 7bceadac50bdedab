"""topk_ragged_static (no workspace, no allocation) against topk_ragged.

Callers that cannot allocate device memory use topk_ragged_static, whose
scratch is a fixed array inside the library. This file runs last so that a
failure here never hides another test; it also passes on its own, in a fresh
process (the first call on the device then sets the array up).
"""
import numpy as np
import pytest

import workloads
from tests.gpu_util import Runner, canonical

pytestmark = pytest.mark.gpu


def _run_static(rn, w):
    torch = rn.torch
    x = torch.from_numpy(w.logits).to(rn.dev)
    ln = torch.from_numpy(w.lengths).to(rn.dev)
    out = torch.full((w.num_rows, w.topk), -7, dtype=torch.int32, device=rn.dev)
    rc = rn.sar.topk_ragged_static(x, w.row_stride, ln, w.num_rows, w.next_n, w.topk, out)
    assert rc == rn.sar.TOPK_OK, rn.sar.topk_status_string(rc)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _same_sets(w, a, b, label):
    for r in range(w.num_rows):
        ca = canonical(w.logits[r], w.lengths[r], a[r])
        cb = canonical(w.logits[r], w.lengths[r], b[r])
        assert ca == cb, f"{label}: row {r} differs between topk_ragged_static and topk_ragged"


def test_static_matches_workspace_entry_point_twice():
    rn = Runner()
    # rows split across CTAs (the scratch holds their group state), then whole rows
    cases = [workloads.make("long_coop", 3), workloads.make("decode_batch", 10), workloads.make("mtp", 4)]
    for call in range(2):
        for w in cases:
            want = rn.run(w.logits, w.lengths, w.topk, w.next_n)
            got = _run_static(rn, w)
            _same_sets(w, got, want, f"call {call} {w.name}")
    # a changed batch through the same scratch
    w = workloads.make("long_coop", 3)
    rng = np.random.default_rng(77)
    w.logits = np.round(rng.standard_normal(w.logits.shape) * 8).astype(np.float32) / 8
    _same_sets(w, _run_static(rn, w), rn.run(w.logits, w.lengths, w.topk, w.next_n), "changed batch")
