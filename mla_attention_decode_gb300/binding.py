"""ctypes binding of libmla_decode.so (argument marshalling only).

The names mirror the C ABI in include/mla_decode.h: ``mla_decode_plan``,
``mla_decode_workspace_bytes``, ``mla_decode_fwd``, ``mla_decode_poll_error``,
``mla_status_string``.  Tensors are passed by device pointer; every step of the
decode runs in the library's CUDA kernels.  The library is loaded on first use;
a missing library raises -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmla_decode.so")

MLA_KV_BF16, MLA_KV_FP8_E4M3, MLA_KV_MXFP4 = 0, 1, 2
KV_DTYPE_CODES = {"bf16": MLA_KV_BF16, "fp8": MLA_KV_FP8_E4M3, "mxfp4": MLA_KV_MXFP4}
MLA_OK = 0
MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED, MLA_ERR_WORKSPACE_TOO_SMALL, MLA_ERR_CUDA = 1, 2, 3, 4
MLA_ERR_DEVICE_INDEX, MLA_ERR_DEVICE_TIMEOUT, MLA_ERR_NO_DEVICE = 5, 6, 7
SM_SCALE = 1.0 / 24.0


class MLAError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {mla_status_string(status)} (status {status})")


class mla_plan(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("kv_dtype", ctypes.c_int32), ("total_kv", ctypes.c_int32),
                ("chunk_tokens", ctypes.c_int32), ("max_splits", ctypes.c_int32), ("num_work", ctypes.c_int32),
                ("grid", ctypes.c_int32), ("num_sms", ctypes.c_int32), ("splits_max", ctypes.c_int32),
                ("tile_tokens", ctypes.c_int32), ("units_per_cta", ctypes.c_int32),
                ("schedule", ctypes.c_int32), ("total_tiles", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("num_pages", ctypes.c_int32), ("unit_cost", ctypes.c_int32), ("q_len", ctypes.c_int32),
                ("tokens_fused", ctypes.c_int32), ("mx_scores", ctypes.c_int32),
                ("late_tiles", ctypes.c_int32),
                ("first_row", ctypes.c_int32 * 256)]

    def as_dict(self) -> dict:
        return {k: getattr(self, k) for k, _ in self._fields_ if k != "first_row"}


_lock = threading.Lock()
_lib: ctypes.CDLL | None = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads (once) and binds the shared library; raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with `python -m mla_attention_decode_gb300.build` "
                               "(the CUDA library is required; there is no CPU fallback)")
        lib = ctypes.CDLL(path)
        P, i32 = ctypes.c_void_p, ctypes.c_int32
        lib.mla_decode_plan.argtypes = [P, i32, i32, i32, i32, ctypes.POINTER(mla_plan)]
        lib.mla_decode_plan.restype = ctypes.c_int
        lib.mla_decode_workspace_bytes.argtypes = [ctypes.POINTER(mla_plan)]
        lib.mla_decode_workspace_bytes.restype = ctypes.c_size_t
        lib.mla_decode_fwd.argtypes = [P, P, P, i32, P, P, P, P, ctypes.c_float, ctypes.POINTER(mla_plan), P,
                                       ctypes.c_size_t, P]
        lib.mla_decode_fwd.restype = ctypes.c_int
        lib.mla_decode_plan_multi.argtypes = [P, i32, i32, i32, i32, i32, ctypes.POINTER(mla_plan)]
        lib.mla_decode_plan_multi.restype = ctypes.c_int
        lib.mla_decode_plan_paged.argtypes = [P, P, i32, i32, i32, i32, i32, i32, ctypes.POINTER(mla_plan)]
        lib.mla_decode_plan_paged.restype = ctypes.c_int
        lib.mla_decode_fwd_paged.argtypes = [P, P, P, i32, P, P, P, P, P, P, ctypes.c_float,
                                             ctypes.POINTER(mla_plan), P, ctypes.c_size_t, P]
        lib.mla_decode_fwd_paged.restype = ctypes.c_int
        lib.mla_decode_split.argtypes = list(lib.mla_decode_fwd.argtypes)
        lib.mla_decode_split.restype = ctypes.c_int
        lib.mla_decode_combine.argtypes = [P, P, ctypes.POINTER(mla_plan), P, ctypes.c_size_t, P]
        lib.mla_decode_combine.restype = ctypes.c_int
        lib.mla_decode_poll_error.argtypes = [P, P]
        lib.mla_decode_poll_error.restype = ctypes.c_int
        lib.mla_status_string.argtypes = [ctypes.c_int]
        lib.mla_status_string.restype = ctypes.c_char_p
        lib.mla_decode_version.argtypes = []
        lib.mla_decode_version.restype = ctypes.c_char_p
        _lib = lib
        return lib


def mla_status_string(status: int) -> str:
    return load_library().mla_status_string(int(status)).decode()


def mla_decode_version() -> str:
    return load_library().mla_decode_version().decode()


def _dtype_code(kv_dtype) -> int:
    return KV_DTYPE_CODES[kv_dtype] if isinstance(kv_dtype, str) else int(kv_dtype)


def mla_decode_plan(kv_indptr_host, kv_dtype, num_sms: int = 0, num_splits: int = 0) -> mla_plan:
    """Host planner.  ``kv_indptr_host``: CPU int32 tensor / sequence of length batch+1."""
    ind = torch.as_tensor(kv_indptr_host, dtype=torch.int32, device="cpu").contiguous()
    plan = mla_plan()
    rc = load_library().mla_decode_plan(ctypes.c_void_p(ind.data_ptr()), int(ind.numel() - 1),
                                        _dtype_code(kv_dtype), int(num_sms), int(num_splits), ctypes.byref(plan))
    if rc != MLA_OK:
        raise MLAError(rc, "mla_decode_plan")
    return plan


def mla_decode_plan_multi(kv_indptr_host, q_len: int, kv_dtype, num_sms: int = 0, num_splits: int = 0) -> mla_plan:
    """Host planner for q_len query tokens per sequence (see mla_decode.h)."""
    ind = torch.as_tensor(kv_indptr_host, dtype=torch.int32, device="cpu").contiguous()
    plan = mla_plan()
    rc = load_library().mla_decode_plan_multi(ctypes.c_void_p(ind.data_ptr()), int(ind.numel() - 1), int(q_len),
                                              _dtype_code(kv_dtype), int(num_sms), int(num_splits),
                                              ctypes.byref(plan))
    if rc != MLA_OK:
        raise MLAError(rc, "mla_decode_plan_multi")
    return plan


def mla_decode_plan_paged(kv_page_indptr_host, kv_last_page_len_host, page_size: int, num_pages: int, kv_dtype,
                          num_sms: int = 0, num_splits: int = 0) -> mla_plan:
    """Host planner for a paged cache (see mla_decode.h): page-counted indptr
    [batch+1] and last-page lengths [batch] as CPU int32 data."""
    ind = torch.as_tensor(kv_page_indptr_host, dtype=torch.int32, device="cpu").contiguous()
    last = torch.as_tensor(kv_last_page_len_host, dtype=torch.int32, device="cpu").contiguous()
    plan = mla_plan()
    rc = load_library().mla_decode_plan_paged(ctypes.c_void_p(ind.data_ptr()), ctypes.c_void_p(last.data_ptr()),
                                              int(ind.numel() - 1), int(page_size), int(num_pages),
                                              _dtype_code(kv_dtype), int(num_sms), int(num_splits),
                                              ctypes.byref(plan))
    if rc != MLA_OK:
        raise MLAError(rc, "mla_decode_plan_paged")
    return plan


def mla_decode_workspace_bytes(plan: mla_plan) -> int:
    return int(load_library().mla_decode_workspace_bytes(ctypes.byref(plan)))


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def mla_decode_fwd(q, kv, kv_scale, kv_indptr, qo_indptr, out, lse, plan: mla_plan, workspace,
                   sm_scale: float = SM_SCALE, scale_stride: int = 0, stream=None) -> None:
    """Enqueues one decode on ``stream`` (default: torch's current stream).  All
    tensors are CUDA tensors; ``workspace`` is a uint8 tensor of at least
    ``mla_decode_workspace_bytes(plan)`` bytes."""
    if stream is None:
        stream = torch.cuda.current_stream(kv.device)  # q may be pinned host memory
    handle = ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))
    rc = load_library().mla_decode_fwd(_ptr(q), _ptr(kv), _ptr(kv_scale), int(scale_stride), _ptr(kv_indptr),
                                       _ptr(qo_indptr), _ptr(out), _ptr(lse), float(sm_scale), ctypes.byref(plan),
                                       _ptr(workspace), int(workspace.numel() * workspace.element_size()), handle)
    if rc != MLA_OK:
        raise MLAError(rc, "mla_decode_fwd")


def mla_decode_fwd_paged(q, kv_pages, kv_scale, kv_page_indptr, kv_indices, kv_last_page_len, qo_indptr, out, lse,
                         plan: mla_plan, workspace, sm_scale: float = SM_SCALE, scale_stride: int = 0,
                         stream=None) -> None:
    """One decode over a paged cache (plan from mla_decode_plan_paged)."""
    rc = load_library().mla_decode_fwd_paged(_ptr(q), _ptr(kv_pages), _ptr(kv_scale), int(scale_stride),
                                             _ptr(kv_page_indptr), _ptr(kv_indices), _ptr(kv_last_page_len),
                                             _ptr(qo_indptr), _ptr(out), _ptr(lse), float(sm_scale),
                                             ctypes.byref(plan), _ptr(workspace),
                                             int(workspace.numel() * workspace.element_size()),
                                             _stream_handle(stream, kv_pages.device))
    if rc != MLA_OK:
        raise MLAError(rc, "mla_decode_fwd_paged")


def _stream_handle(stream, device) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def mla_decode_split(q, kv, kv_scale, kv_indptr, qo_indptr, out, lse, plan: mla_plan, workspace,
                     sm_scale: float = SM_SCALE, scale_stride: int = 0, stream=None) -> None:
    """Split stage only (see mla_decode.h)."""
    rc = load_library().mla_decode_split(_ptr(q), _ptr(kv), _ptr(kv_scale), int(scale_stride), _ptr(kv_indptr),
                                         _ptr(qo_indptr), _ptr(out), _ptr(lse), float(sm_scale),
                                         ctypes.byref(plan), _ptr(workspace),
                                         int(workspace.numel() * workspace.element_size()),
                                         _stream_handle(stream, kv.device))
    if rc != MLA_OK:
        raise MLAError(rc, "mla_decode_split")


def mla_decode_combine(out, lse, plan: mla_plan, workspace, stream=None) -> None:
    """Combine stage only (see mla_decode.h)."""
    rc = load_library().mla_decode_combine(_ptr(out), _ptr(lse), ctypes.byref(plan), _ptr(workspace),
                                           int(workspace.numel() * workspace.element_size()),
                                           _stream_handle(stream, out.device))
    if rc != MLA_OK:
        raise MLAError(rc, "mla_decode_combine")


def mla_decode_poll_error(workspace, stream=None) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(workspace.device)
    return int(load_library().mla_decode_poll_error(_ptr(workspace), ctypes.c_void_p(stream.cuda_stream)))


MLA_STATIC_WORKSPACE_BYTES = 16 << 20


def mla_decode_fwd_static(q, kv, kv_scale, kv_indptr, qo_indptr, out, lse, plan: mla_plan, device_error=None,
                          sm_scale: float = SM_SCALE, scale_stride: int = 0, stream=None) -> None:
    """mla_decode_fwd without a caller workspace: the library's own device array
    of MLA_STATIC_WORKSPACE_BYTES is used (for callers that cannot allocate).
    ``device_error``: optional int32 CUDA tensor of one element that receives
    the call's device error word.  Calls that overlap on the GPU race."""
    lib = load_library()
    fn = lib.mla_decode_fwd_static
    if fn.argtypes is None:
        P, i32 = ctypes.c_void_p, ctypes.c_int32
        fn.argtypes = [P, P, P, i32, P, P, P, P, ctypes.c_float, ctypes.POINTER(mla_plan), P, P]
        fn.restype = ctypes.c_int
    rc = fn(_ptr(q), _ptr(kv), _ptr(kv_scale), int(scale_stride), _ptr(kv_indptr), _ptr(qo_indptr), _ptr(out),
            _ptr(lse), float(sm_scale), ctypes.byref(plan), _ptr(device_error), _stream_handle(stream, kv.device))
    if rc != MLA_OK:
        raise MLAError(rc, "mla_decode_fwd_static")


class MLADecoder:
    """Plan + workspace for one batch layout; call it with device tensors.

    The workspace is allocated once here (torch device memory) and zeroed; the
    library itself never allocates.  ``q_len > 1``: that many query tokens per
    sequence (rows ``qo_indptr[b] + i``, output rows ``b * q_len + i``); e4m3 KV
    with ``q_len == 2`` gets the single-pass plan (``plan.tokens_fused == 2``).
    ``mx_block_scaled``: MXFP4 scores from block-scaled MMAs on the e2m1 tile
    (``plan.mx_scores = 1``) instead of the e4m3 copy."""

    def __init__(self, kv_indptr_host, kv_dtype, device="cuda", num_sms: int = 0, num_splits: int = 0,
                 q_len: int = 1, mx_block_scaled: bool = False):
        self.kv_dtype = _dtype_code(kv_dtype)
        if q_len > 1:
            self.plan = mla_decode_plan_multi(kv_indptr_host, q_len, self.kv_dtype, num_sms, num_splits)
        else:
            self.plan = mla_decode_plan(kv_indptr_host, self.kv_dtype, num_sms, num_splits)
        if mx_block_scaled:
            self.plan.mx_scores = 1
        nbytes = max(256, mla_decode_workspace_bytes(self.plan))
        self.workspace = torch.zeros(nbytes, dtype=torch.uint8, device=device)

    def __call__(self, q, kv, kv_indptr, qo_indptr, kv_scale=None, out=None, lse=None,
                 sm_scale: float = SM_SCALE, stream=None):
        batch = self.plan.batch
        if out is None:
            out = torch.empty(batch, 16, 512, dtype=torch.bfloat16, device=self.workspace.device)
        if lse is None:
            lse = torch.empty(batch, 16, dtype=torch.float32, device=self.workspace.device)
        scale_stride = int(kv_scale.stride(0)) if (self.kv_dtype == MLA_KV_MXFP4 and kv_scale is not None) else 0
        mla_decode_fwd(q, kv, kv_scale, kv_indptr, qo_indptr, out, lse, self.plan, self.workspace,
                       sm_scale=sm_scale, scale_stride=scale_stride, stream=stream)
        return out, lse

    def poll_error(self, stream=None) -> int:
        return mla_decode_poll_error(self.workspace, stream)


class PagedMLADecoder:
    """Plan + workspace for one paged batch layout (see mla_decode_plan_paged)."""

    def __init__(self, kv_page_indptr_host, kv_last_page_len_host, page_size: int, num_pages: int, kv_dtype,
                 device="cuda", num_sms: int = 0, num_splits: int = 0, mx_block_scaled: bool = False):
        self.kv_dtype = _dtype_code(kv_dtype)
        self.plan = mla_decode_plan_paged(kv_page_indptr_host, kv_last_page_len_host, page_size, num_pages,
                                          self.kv_dtype, num_sms, num_splits)
        if mx_block_scaled:
            self.plan.mx_scores = 1
        nbytes = max(256, mla_decode_workspace_bytes(self.plan))
        self.workspace = torch.zeros(nbytes, dtype=torch.uint8, device=device)

    def __call__(self, q, kv_pages, kv_page_indptr, kv_indices, kv_last_page_len, qo_indptr, kv_scale=None,
                 out=None, lse=None, sm_scale: float = SM_SCALE, stream=None):
        batch = self.plan.batch
        if out is None:
            out = torch.empty(batch, 16, 512, dtype=torch.bfloat16, device=self.workspace.device)
        if lse is None:
            lse = torch.empty(batch, 16, dtype=torch.float32, device=self.workspace.device)
        scale_stride = int(kv_scale.stride(0)) if (self.kv_dtype == MLA_KV_MXFP4 and kv_scale is not None) else 0
        mla_decode_fwd_paged(q, kv_pages, kv_scale, kv_page_indptr, kv_indices, kv_last_page_len, qo_indptr, out,
                             lse, self.plan, self.workspace, sm_scale=sm_scale, scale_stride=scale_stride,
                             stream=stream)
        return out, lse

    def poll_error(self, stream=None) -> int:
        return mla_decode_poll_error(self.workspace, stream)


class PackedBuffers:
    """Several tensors laid out in one pinned host buffer and one device buffer
    (256-byte aligned offsets), so that moving all of them takes one copy each
    way.  ``specs``: list of (name, shape, dtype).  ``host[name]`` and
    ``dev[name]`` are views into the two buffers."""

    def __init__(self, specs, device):
        self.layout = {}
        off = 0
        for name, shape, dtype in specs:
            n = 1
            for x in shape:
                n *= int(x)
            n *= torch.empty((), dtype=dtype).element_size()
            self.layout[name] = (off, tuple(shape), dtype, n)
            off = (off + n + 255) // 256 * 256
        self.nbytes = max(off, 256)
        self.host_bytes = torch.empty(self.nbytes, dtype=torch.uint8).pin_memory()
        self.dev_bytes = torch.empty(self.nbytes, dtype=torch.uint8, device=device)
        self.host = {k: self._view(self.host_bytes, *v) for k, v in self.layout.items()}
        self.dev = {k: self._view(self.dev_bytes, *v) for k, v in self.layout.items()}

    @staticmethod
    def _view(buf, off, shape, dtype, n):
        return buf[off:off + n].view(dtype).view(shape)

    def to_device(self, stream=None):
        """One host-to-device copy of the whole buffer on ``stream`` (asynchronous)."""
        with torch.cuda.stream(stream) if stream is not None else _nullcontext():
            self.dev_bytes.copy_(self.host_bytes, non_blocking=True)

    def to_host(self, stream=None):
        """One device-to-host copy of the whole buffer on ``stream`` (asynchronous)."""
        with torch.cuda.stream(stream) if stream is not None else _nullcontext():
            self.host_bytes.copy_(self.dev_bytes, non_blocking=True)


class _nullcontext:
    def __enter__(self):
        return None

    def __exit__(self, *a):
        return False
