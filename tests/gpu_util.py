"""Helpers for the GPU parity tests: run libtopk on host arrays and compare with the oracle."""
from __future__ import annotations

import numpy as np

import oracle


def require_cuda():
    import torch

    if not torch.cuda.is_available():
        raise RuntimeError("these tests need a CUDA GPU")
    from sparse_attention_row_gb300 import build

    build.build_library()


def canonical(x_row: np.ndarray, length: int, sel: np.ndarray) -> list[int]:
    """Sorts a selected index set by (value desc, index asc), -1 entries last.

    Fails if an index is outside [0, length) or repeated, since such a result
    can never match the oracle.
    """
    length = max(0, min(int(length), x_row.shape[0]))
    sel = np.asarray(sel, dtype=np.int64)
    valid = sel[sel >= 0]
    assert np.all(sel >= -1), f"index below -1: {sel.min()}"
    assert np.all(valid < length), f"index {valid.max()} beyond length {length}"
    assert len(np.unique(valid)) == len(valid), "repeated index"
    order = np.lexsort((valid, -x_row[valid].astype(np.float64)))
    out = valid[order].tolist()
    return out + [-1] * (len(sel) - len(out))


def assert_matches_oracle(x: np.ndarray, lengths: np.ndarray, got: np.ndarray, topk: int,
                          next_n: int = 1, want: np.ndarray | None = None, label: str = ""):
    if want is None:
        want, _ = oracle.topk_ragged(x, lengths, topk, next_n=next_n)
    bad = []
    for r in range(x.shape[0]):
        c = canonical(x[r], lengths[r], got[r])
        if c != want[r].tolist():
            bad.append(r)
            if len(bad) > 3:
                break
    if bad:
        r = bad[0]
        c = canonical(x[r], lengths[r], got[r])
        w = want[r].tolist()
        first = next(i for i in range(len(w)) if c[i] != w[i])
        raise AssertionError(
            f"{label}: rows {bad} differ from the oracle; row {r} (len {int(lengths[r])}) first "
            f"difference at rank {first}: gpu {c[first:first + 4]} oracle {w[first:first + 4]}")


class Runner:
    """Runs libtopk on host arrays through the C ABI, with torch for device memory."""

    def __init__(self, device: int = 0):
        import torch

        import sparse_attention_row_gb300 as sar

        require_cuda()
        self.torch = torch
        self.sar = sar
        self.dev = torch.device("cuda", device)
        self.sel = sar.Selector(device)

    def to_dev(self, x: np.ndarray, pad_front: int = 0):
        """Copies logits to the device; pad_front elements shift the base address."""
        flat = self.torch.empty(x.size + pad_front + 4, dtype=self.torch.float32, device=self.dev)
        flat[pad_front:pad_front + x.size] = self.torch.from_numpy(np.ascontiguousarray(x).reshape(-1)).to(self.dev)
        return flat, flat[pad_front:]

    def run(self, x: np.ndarray, lengths: np.ndarray, topk: int, next_n: int = 1,
            options=None, pad_front: int = 0, check_status: bool = True) -> np.ndarray:
        torch = self.torch
        sar = self.sar
        num_rows, stride = x.shape
        _, xd = self.to_dev(x, pad_front)
        ln = torch.from_numpy(np.ascontiguousarray(lengths, dtype=np.int32)).to(self.dev)
        out = torch.full((num_rows, topk), -7, dtype=torch.int32, device=self.dev)
        rc = sar.topk_ragged_ex(xd, stride, ln, num_rows, next_n, topk, out, self.sel.workspace,
                                None, options)
        assert rc == sar.TOPK_OK, sar.topk_status_string(rc)
        torch.cuda.synchronize()
        if check_status:
            st = self.sel.status()
            assert st & ~sar.TOPK_DEV_LENGTH_CLAMPED == 0, f"device status {st:#x}"
        return out.cpu().numpy()

    def workspace_clean(self) -> bool:
        """True if every workspace byte after the status word is zero."""
        self.torch.cuda.synchronize()
        ws = self.sel.workspace.cpu().numpy()
        return not ws[256:].any()

    def options(self, **kw):
        o = self.sar.TopkOptions()
        for k, v in kw.items():
            setattr(o, k, v)
        return o
