"""Python binding of libtopk (ragged per-row top-K on GB300).

Argument marshalling only: every function here forwards to the C ABI declared
in ``include/libtopk.h`` with the same name; all computation runs in the CUDA
kernels of ``libtopk.so``. Tensor arguments may be torch tensors (their
``data_ptr()`` is passed) or raw integer device addresses. PyTorch serves only
as the provider of device memory and streams.

If ``libtopk.so`` has not been built this module raises on first use; there is
no CPU or PyTorch fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "TOPK_OK", "TopkError", "TopkOptions", "TopkDeviceProps", "TopkPlan",
    "topk_workspace_size", "topk_workspace_init", "topk_ragged", "topk_ragged_ex", "topk_ragged_static",
    "topk_ragged_strided", "topk_gather_sort",
    "topk_get_status", "topk_status_string", "topk_query_device", "topk_make_plan",
    "library_path", "Selector",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libtopk.so")
_lock = threading.Lock()
_lib = None

TOPK_OK = 0
TOPK_ERR_INVALID_ARG = 1
TOPK_ERR_UNSUPPORTED_TOPK = 2
TOPK_ERR_MISALIGNED = 3
TOPK_ERR_WORKSPACE_TOO_SMALL = 4
TOPK_ERR_CUDA = 5
TOPK_ERR_BARRIER_TIMEOUT = 6
TOPK_ERR_LENGTH_CLAMPED = 7
TOPK_ERR_PLAN = 8

TOPK_MERGE_AUTO = 0
TOPK_MERGE_WORKSPACE = 1
TOPK_MERGE_CLUSTER = 2

TOPK_SHAPE_AUTO = 0
TOPK_SHAPE_WIDE = 1
TOPK_SHAPE_PAIR = 2
TOPK_SHAPE_SMALL = 3
TOPK_SHAPE_SHORT = 4

TOPK_DEV_LENGTH_CLAMPED = 0x1
TOPK_DEV_BARRIER_TIMEOUT = 0x2
TOPK_DEV_STAGE_TIMEOUT = 0x4
TOPK_DEV_WORKSPACE_DIRTY = 0x8

EXPORTED = ("topk_workspace_size", "topk_workspace_init", "topk_ragged", "topk_ragged_ex", "topk_ragged_static",
            "topk_ragged_strided", "topk_gather_sort", "topk_get_status", "topk_status_string",
            "topk_query_device", "topk_make_plan")


class TopkError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {topk_status_string(code)} (code {code})")


class TopkOptions(ctypes.Structure):
    _fields_ = [("force_ctas_per_group", ctypes.c_int),
                ("long_row_threshold", ctypes.c_int64),
                ("barrier_timeout_us", ctypes.c_uint32),
                ("inject_skip_arrival", ctypes.c_int),
                ("workspace_bytes", ctypes.c_size_t),
                ("max_ctas", ctypes.c_int),
                ("merge", ctypes.c_int),
                ("shape", ctypes.c_int),
                ("dependent_launch", ctypes.c_int)]


class TopkDeviceProps(ctypes.Structure):
    _fields_ = [("num_sms", ctypes.c_int),
                ("max_smem_optin", ctypes.c_int),
                ("smem_per_cta", ctypes.c_int),
                ("ctas_per_sm", ctypes.c_int),
                ("cluster_groups", ctypes.c_int * 9),
                ("pair_smem_per_cta", ctypes.c_int),
                ("pair_ctas_per_sm", ctypes.c_int),
                ("small_smem_per_cta", ctypes.c_int),
                ("small_ctas_per_sm", ctypes.c_int),
                ("short_smem_per_cta", ctypes.c_int),
                ("short_ctas_per_sm", ctypes.c_int),
                ("short_cluster_groups", ctypes.c_int * 9),
                ("short16_smem_per_cta", ctypes.c_int),
                ("short16_ctas_per_sm", ctypes.c_int),
                ("short16_cluster_groups", ctypes.c_int * 9)]


class TopkPlan(ctypes.Structure):
    _fields_ = [("ctas_per_group", ctypes.c_int),
                ("num_groups", ctypes.c_int),
                ("grid", ctypes.c_int),
                ("threads", ctypes.c_int),
                ("smem_bytes", ctypes.c_int),
                ("cooperative", ctypes.c_int),
                ("cluster", ctypes.c_int),
                ("shape", ctypes.c_int)]


def library_path() -> str:
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is missing: build it with `python -m sparse_attention_row_gb300.build` "
                "(or __graft_entry__.build()); there is no fallback implementation")
        lib = ctypes.CDLL(_LIB_PATH)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.topk_workspace_size.restype = ctypes.c_size_t
        lib.topk_workspace_size.argtypes = [i32, i64, i64, i32, i32]
        lib.topk_workspace_init.restype = i32
        lib.topk_workspace_init.argtypes = [vp, ctypes.c_size_t, vp]
        lib.topk_ragged.restype = i32
        lib.topk_ragged.argtypes = [vp, i64, vp, i64, i32, i32, vp, vp, vp]
        lib.topk_ragged_ex.restype = i32
        lib.topk_ragged_ex.argtypes = [vp, i64, vp, i64, i32, i32, vp, vp, vp,
                                       ctypes.POINTER(TopkOptions)]
        lib.topk_ragged_strided.restype = i32
        lib.topk_ragged_strided.argtypes = [vp, i64, i64, i64, vp, i64, i32, i32, vp, vp, vp,
                                            ctypes.POINTER(TopkOptions)]
        lib.topk_gather_sort.restype = i32
        lib.topk_gather_sort.argtypes = [vp, i64, i64, i64, i64, i32, vp, vp, i32, vp]
        lib.topk_ragged_static.restype = i32
        lib.topk_ragged_static.argtypes = [vp, i64, vp, i64, i32, i32, vp, vp]
        lib.topk_get_status.restype = i32
        lib.topk_get_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint32)]
        lib.topk_status_string.restype = ctypes.c_char_p
        lib.topk_status_string.argtypes = [i32]
        lib.topk_query_device.restype = i32
        lib.topk_query_device.argtypes = [i32, ctypes.POINTER(TopkDeviceProps)]
        lib.topk_make_plan.restype = i32
        lib.topk_make_plan.argtypes = [ctypes.POINTER(TopkDeviceProps), i64, i64, i32, i32,
                                       ctypes.POINTER(TopkOptions), ctypes.POINTER(TopkPlan)]
        _lib = lib
        return lib


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return int(x.data_ptr())
    raise TypeError(f"expected a tensor or an integer address, got {type(x).__name__}")


def _stream(stream) -> int | None:
    if stream is None:
        try:
            import torch

            if torch.cuda.is_available():
                return int(torch.cuda.current_stream().cuda_stream)
        except ImportError:
            pass
        return None
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def topk_status_string(code: int) -> str:
    return _load().topk_status_string(int(code)).decode()


def topk_workspace_size(device: int, num_rows: int = 0, row_stride: int = 1, next_n: int = 1,
                        topk: int = 2048) -> int:
    return int(_load().topk_workspace_size(device, num_rows, row_stride, next_n, topk))


def topk_workspace_init(workspace, nbytes: int, stream=None) -> int:
    return int(_load().topk_workspace_init(_ptr(workspace), nbytes, _stream(stream)))


def topk_ragged(logits, row_stride: int, lengths, num_rows: int, next_n: int, topk: int, out_idx,
                workspace, stream=None) -> int:
    return int(_load().topk_ragged(_ptr(logits), row_stride, _ptr(lengths), num_rows, next_n, topk,
                                   _ptr(out_idx), _ptr(workspace), _stream(stream)))


def topk_ragged_ex(logits, row_stride: int, lengths, num_rows: int, next_n: int, topk: int, out_idx,
                   workspace, stream=None, options: TopkOptions | None = None) -> int:
    opt = ctypes.byref(options) if options is not None else None
    return int(_load().topk_ragged_ex(_ptr(logits), row_stride, _ptr(lengths), num_rows, next_n,
                                      topk, _ptr(out_idx), _ptr(workspace), _stream(stream), opt))


def topk_ragged_strided(logits, row_stride: int, col_stride: int, max_len: int, lengths, num_rows: int,
                        next_n: int, topk: int, out_idx, workspace, stream=None,
                        options: TopkOptions | None = None) -> int:
    """topk_ragged over a strided view: element (r, i) at logits[r * row_stride + i * col_stride]."""
    opt = ctypes.byref(options) if options is not None else None
    return int(_load().topk_ragged_strided(_ptr(logits), row_stride, col_stride, max_len, _ptr(lengths),
                                           num_rows, next_n, topk, _ptr(out_idx), _ptr(workspace),
                                           _stream(stream), opt))


def topk_gather_sort(logits, row_stride: int, col_stride: int, max_len: int, num_rows: int, topk: int,
                     out_idx, out_val=None, sort: bool = True, stream=None) -> int:
    """Values of the selected indices (if out_val is given) and, with sort, rows ordered by
    value descending then index ascending, -1 last."""
    return int(_load().topk_gather_sort(_ptr(logits), row_stride, col_stride, max_len, num_rows, topk,
                                        _ptr(out_idx), _ptr(out_val), 1 if sort else 0, _stream(stream)))


def topk_ragged_static(logits, row_stride: int, lengths, num_rows: int, next_n: int, topk: int,
                       out_idx, stream=None) -> int:
    """topk_ragged for callers that cannot allocate: no workspace argument."""
    return int(_load().topk_ragged_static(_ptr(logits), row_stride, _ptr(lengths), num_rows, next_n,
                                          topk, _ptr(out_idx), _stream(stream)))


def topk_get_status(workspace, stream=None) -> tuple[int, int]:
    """Returns (code, device status bits); synchronises the stream."""
    word = ctypes.c_uint32(0)
    rc = _load().topk_get_status(_ptr(workspace), _stream(stream), ctypes.byref(word))
    return int(rc), int(word.value)


def topk_query_device(device: int) -> TopkDeviceProps:
    props = TopkDeviceProps()
    rc = _load().topk_query_device(device, ctypes.byref(props))
    if rc != TOPK_OK:
        raise TopkError(rc, "topk_query_device")
    return props


def topk_make_plan(props: TopkDeviceProps, num_rows: int, row_stride: int, next_n: int, topk: int,
                   options: TopkOptions | None = None) -> tuple[int, TopkPlan]:
    plan = TopkPlan()
    opt = ctypes.byref(options) if options is not None else None
    rc = _load().topk_make_plan(ctypes.byref(props), num_rows, row_stride, next_n, topk, opt,
                                ctypes.byref(plan))
    return int(rc), plan


class Selector:
    """Owns one workspace on one device and runs calls on a stream.

    Uses torch only to allocate the workspace and the output. Calls that may
    overlap on the GPU need separate Selectors (separate workspaces).
    """

    def __init__(self, device: int = 0):
        import torch

        self.device = device
        self.nbytes = topk_workspace_size(device)
        if self.nbytes == 0:
            raise TopkError(TOPK_ERR_CUDA, "topk_workspace_size")
        self.workspace = torch.empty(self.nbytes, dtype=torch.uint8, device=f"cuda:{device}")
        rc = topk_workspace_init(self.workspace, self.nbytes)
        if rc != TOPK_OK:
            raise TopkError(rc, "topk_workspace_init")

    def __call__(self, logits, lengths, topk: int, next_n: int | None = None, out=None, stream=None,
                 options: TopkOptions | None = None, sort: bool = False, values: bool = False):
        """Top-K indices of every row of a float32 [num_rows, max_len] tensor (any strides);
        with values=True also their values (returns (indices, values)), with sort=True each row
        ordered by value descending then index ascending, -1 last.

        lengths: int32, [num_rows], or [num_rows / next_n, next_n] for MTP, in which
        case next_n is taken from its second dimension (as the pages' launcher does).
        """
        import torch

        if logits.dtype != torch.float32 or logits.dim() != 2:
            raise ValueError("logits must be a float32 [num_rows, max_len] tensor")
        if lengths.dtype != torch.int32 or not lengths.is_contiguous() or lengths.dim() not in (1, 2):
            raise ValueError("lengths must be a contiguous int32 tensor with 1 or 2 dimensions")
        if next_n is None:
            next_n = lengths.shape[1] if lengths.dim() == 2 else 1
        num_rows, max_len = logits.shape
        if lengths.numel() != num_rows:
            raise ValueError("lengths must hold one length per row")
        if out is None:
            out = torch.empty((num_rows, topk), dtype=torch.int32, device=logits.device)
        # contiguous rows (stride(1) == 1) take the bulk-copy path inside the library
        rc = topk_ragged_strided(logits, logits.stride(0), logits.stride(1), max_len, lengths, num_rows,
                                 next_n, topk, out, self.workspace, stream, options)
        if rc != TOPK_OK:
            raise TopkError(rc, "topk_ragged")
        if not (sort or values):
            return out
        val = torch.empty((num_rows, topk), dtype=torch.float32, device=logits.device) if values else None
        rc = topk_gather_sort(logits, logits.stride(0), logits.stride(1), max_len, num_rows, topk, out, val,
                              sort, stream)
        if rc != TOPK_OK:
            raise TopkError(rc, "topk_gather_sort")
        return (out, val) if values else out

    def status(self, stream=None) -> int:
        rc, word = topk_get_status(self.workspace, stream)
        if rc != TOPK_OK:
            raise TopkError(rc, "topk_get_status")
        return word

    def reset(self, stream=None) -> None:
        rc = topk_workspace_init(self.workspace, self.nbytes, stream)
        if rc != TOPK_OK:
            raise TopkError(rc, "topk_workspace_init")
