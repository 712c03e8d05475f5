"""ctypes binding of libep.so: argument marshalling only.

Every step of layout, dispatch and combine runs in the library's CUDA
kernels; this module only turns torch tensors into pointers and the current
torch stream into a ``cudaStream_t``, allocates output tensors when asked,
and exposes the handle's device arrays as zero-copy torch views.  There is no
CPU fallback: if ``libep.so`` is missing or cannot be loaded, every call
raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libep.so")

EP_OK = 0
EP_ERR_INVALID_ARG = 1
EP_ERR_UNSUPPORTED = 2
EP_ERR_BAD_TOPK_IDX = 3
EP_ERR_CUDA = 4
EP_ERR_OOM = 5
EP_ERR_TIMEOUT = 6
EP_ERR_OVERFLOW = 7
EP_ERRBIT_BAD_TOPK_IDX = 1
EP_ERRBIT_OVERFLOW = 2
EP_ERRBIT_TIMEOUT = 4
EP_ABI_VERSION = 3


class EpError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


class EpConfigC(ctypes.Structure):
    _fields_ = [
        ("num_tokens", ctypes.c_int32),
        ("num_topk", ctypes.c_int32),
        ("num_experts", ctypes.c_int32),
        ("num_ranks", ctypes.c_int32),
        ("hidden", ctypes.c_int32),
        ("num_max_tokens_per_rank", ctypes.c_int32),
        ("expert_alignment", ctypes.c_int32),
        ("topk_idx_is_int64", ctypes.c_int32),
        ("do_expand", ctypes.c_uint8),
        ("do_zero_padding", ctypes.c_uint8),
        ("do_cpu_sync", ctypes.c_uint8),
        ("use_fp8", ctypes.c_uint8),
        ("use_tma_aligned_col_major_sf", ctypes.c_uint8),
        ("fixed_capacity", ctypes.c_uint8),
        ("reserved0", ctypes.c_uint8 * 2),
        ("num_sms", ctypes.c_int32),
        ("cpu_sync_timeout_ms", ctypes.c_int32),
    ]


_P32 = ctypes.c_void_p


class EpLayoutInfoC(ctypes.Structure):
    _fields_ = [
        ("num_recv_tokens", ctypes.c_int64),
        ("num_expanded_tokens", ctypes.c_int64),
        ("rows_alloc", ctypes.c_int64),
        ("sf_numel", ctypes.c_int64),
        ("sf_token_stride", ctypes.c_int64),
        ("sf_hidden_stride", ctypes.c_int64),
        ("topk_idx", _P32),
        ("cnt_expert", _P32),
        ("cnt_expert_aligned", _P32),
        ("psum_expert", _P32),
        ("cnt_rank", _P32),
        ("psum_rank", _P32),
        ("psum_rank_src", _P32),
        ("dst_buffer_slot_idx", _P32),
        ("recv_src_metadata", _P32),
        ("is_token_in_rank", _P32),
        ("totals", _P32),
        ("error_word", _P32),
        ("meta_rows", ctypes.c_int64),
        ("expert_capacity", ctypes.c_int64),
        ("sf_expert_stride", ctypes.c_int64),
        ("layout_kernels", ctypes.c_int32),
        ("reserved1", ctypes.c_int32),
    ]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libep.so once; raise if it is missing (no fallback exists)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    lib.ep_layout.argtypes = [ctypes.POINTER(EpConfigC), vp, vp, ctypes.POINTER(vp),
                              ctypes.POINTER(EpLayoutInfoC)]
    lib.ep_layout.restype = ctypes.c_int
    lib.ep_dispatch.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp]
    lib.ep_dispatch.restype = ctypes.c_int
    lib.ep_combine.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp]
    lib.ep_combine.restype = ctypes.c_int
    lib.ep_dispatch_fp8.argtypes = [vp, vp, vp, i64, i64, vp, vp, vp, vp, vp, vp]
    lib.ep_dispatch_fp8.restype = ctypes.c_int
    lib.ep_dispatch_backward.argtypes = [vp, vp, vp, vp, vp, vp]
    lib.ep_dispatch_backward.restype = ctypes.c_int
    lib.ep_combine_backward.argtypes = [vp, vp, vp, vp]
    lib.ep_combine_backward.restype = ctypes.c_int
    lib.ep_handle_free.argtypes = [vp]
    lib.ep_handle_free.restype = None
    lib.ep_status_string.argtypes = [ctypes.c_int]
    lib.ep_status_string.restype = ctypes.c_char_p
    lib.ep_abi_version.argtypes = []
    lib.ep_abi_version.restype = i32
    lib.ep_validate_config.argtypes = [ctypes.POINTER(EpConfigC)]
    lib.ep_validate_config.restype = ctypes.c_int
    lib.ep_upper_bound_rows.argtypes = [ctypes.POINTER(EpConfigC), ctypes.POINTER(i64)]
    lib.ep_upper_bound_rows.restype = ctypes.c_int
    lib.ep_host_wait_flag.argtypes = [ctypes.POINTER(i32), i32, i32]
    lib.ep_host_wait_flag.restype = ctypes.c_int
    lib.ep_plan_layout.argtypes = [ctypes.POINTER(EpConfigC), ctypes.POINTER(EpLayoutInfoC)]
    lib.ep_plan_layout.restype = ctypes.c_int
    lib.ep_layout_dispatch.argtypes = [ctypes.POINTER(EpConfigC), vp, vp, vp, vp, vp, vp, vp, vp,
                                       ctypes.POINTER(vp), ctypes.POINTER(EpLayoutInfoC)]
    lib.ep_layout_dispatch.restype = ctypes.c_int
    if lib.ep_abi_version() != EP_ABI_VERSION:
        raise RuntimeError("libep.so ABI version does not match this binding")
    _lib = lib
    return lib


def status_string(status: int) -> str:
    try:
        return load_library().ep_status_string(status).decode()
    except RuntimeError:
        return "library not loaded"


def make_config(num_tokens, num_topk, num_experts, num_ranks, hidden, num_max_tokens_per_rank,
                expert_alignment=1, do_expand=False, do_zero_padding=False, do_cpu_sync=True,
                use_fp8=False, use_tma_aligned_col_major_sf=False, num_sms=0,
                cpu_sync_timeout_ms=0, topk_idx_is_int64=True,
                fixed_capacity=False) -> EpConfigC:
    c = EpConfigC()
    c.num_tokens = num_tokens
    c.num_topk = num_topk
    c.num_experts = num_experts
    c.num_ranks = num_ranks
    c.hidden = hidden
    c.num_max_tokens_per_rank = num_max_tokens_per_rank
    c.expert_alignment = expert_alignment
    c.topk_idx_is_int64 = 1 if topk_idx_is_int64 else 0
    c.do_expand = int(bool(do_expand))
    c.do_zero_padding = int(bool(do_zero_padding))
    c.do_cpu_sync = int(bool(do_cpu_sync))
    c.use_fp8 = int(bool(use_fp8))
    c.use_tma_aligned_col_major_sf = int(bool(use_tma_aligned_col_major_sf))
    c.fixed_capacity = int(bool(fixed_capacity))
    c.num_sms = num_sms
    c.cpu_sync_timeout_ms = cpu_sync_timeout_ms
    return c


def validate_config(cfg: EpConfigC) -> int:
    return load_library().ep_validate_config(ctypes.byref(cfg))


def upper_bound_rows(cfg: EpConfigC) -> int:
    rows = ctypes.c_int64(0)
    st = load_library().ep_upper_bound_rows(ctypes.byref(cfg), ctypes.byref(rows))
    if st != EP_OK:
        raise EpError(st, "ep_upper_bound_rows")
    return rows.value


def _stream_ptr(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t: Optional[torch.Tensor], what: str, dtype=None) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise ValueError(f"{what} has dtype {t.dtype}, expected {dtype}")
    return t.data_ptr() if t.numel() > 0 else None


class _DeviceArray:
    """Zero-copy __cuda_array_interface__ view of a device array owned by a handle."""

    def __init__(self, ptr: int, shape, typestr: str, owner):
        self._owner = owner
        self.__cuda_array_interface__ = {
            "shape": tuple(int(s) for s in shape), "typestr": typestr,
            "data": (int(ptr) if ptr else 0, False), "version": 3, "strides": None,
        }


class Handle:
    """Owns an ``ep_handle*``; ``free()`` (or garbage collection) releases it."""

    _ARRAYS = {
        "topk_idx": ("<i4", lambda h: (h.T, h.K)),
        "cnt_expert": ("<i4", lambda h: (h.E,)),
        "cnt_expert_aligned": ("<i4", lambda h: (h.E,)),
        "psum_expert": ("<i4", lambda h: (h.E + 1,)),
        "cnt_rank": ("<i4", lambda h: (h.R,)),
        "psum_rank": ("<i4", lambda h: (h.R + 1,)),
        "psum_rank_src": ("<i4", lambda h: (h.R, h.R + 1)),
        "dst_buffer_slot_idx": ("<i4", lambda h: (h.T, h.K)),
        "recv_src_metadata": ("<i4", lambda h: (h.info.meta_rows, 2)),
        "is_token_in_rank": ("|u1", lambda h: (h.T, h.R)),
        "totals": ("<i4", lambda h: (2,)),
        "error_word": ("<i4", lambda h: (1,)),
    }

    def __init__(self, ptr: int, cfg: EpConfigC, info: EpLayoutInfoC, status: int):
        self._ptr = ptr
        self.cfg = cfg
        self.info = info
        self.status = status
        self.T, self.K, self.E, self.R = cfg.num_tokens, cfg.num_topk, cfg.num_experts, cfg.num_ranks
        self.H = cfg.hidden

    @property
    def ptr(self) -> int:
        if not self._ptr:
            raise RuntimeError("handle already freed")
        return self._ptr

    @property
    def rows_alloc(self) -> int:
        return int(self.info.rows_alloc)

    def tensor(self, name: str) -> torch.Tensor:
        """Zero-copy torch view of one of the handle's device arrays."""
        typestr, shape = self._ARRAYS[name]
        ptr = getattr(self.info, name)
        if not self._ptr:
            raise RuntimeError("handle already freed")
        arr = _DeviceArray(ptr, shape(self), typestr, self)
        if 0 in arr.__cuda_array_interface__["shape"]:
            dt = {"<i4": torch.int32, "|u1": torch.uint8}[typestr]
            return torch.empty(arr.__cuda_array_interface__["shape"], dtype=dt, device="cuda")
        t = torch.as_tensor(arr, device="cuda")
        return t

    def free(self):
        if self._ptr:
            load_library().ep_handle_free(ctypes.c_void_p(self._ptr))
            self._ptr = 0

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


def ep_layout(cfg: EpConfigC, topk_idx: torch.Tensor, stream=None) -> Handle:
    lib = load_library()
    if topk_idx.dtype not in (torch.int64, torch.int32):
        raise ValueError("topk_idx must be int64 or int32")
    if tuple(topk_idx.shape) != (cfg.num_tokens, cfg.num_topk):
        raise ValueError(f"topk_idx shape {tuple(topk_idx.shape)} != "
                         f"({cfg.num_tokens}, {cfg.num_topk})")
    cfg.topk_idx_is_int64 = 1 if topk_idx.dtype == torch.int64 else 0
    p = _ptr(topk_idx, "topk_idx")
    h = ctypes.c_void_p(0)
    info = EpLayoutInfoC()
    st = lib.ep_layout(ctypes.byref(cfg), p, _stream_ptr(stream), ctypes.byref(h),
                       ctypes.byref(info))
    if st not in (EP_OK, EP_ERR_BAD_TOPK_IDX):
        raise EpError(st, "ep_layout")
    cfg_copy = EpConfigC.from_buffer_copy(cfg)
    return Handle(h.value, cfg_copy, info, st)


def _alloc(cfg: EpConfigC, info: EpLayoutInfoC, with_weights: bool, with_idx: bool,
           zero: bool) -> dict:
    rows, H, K = int(info.rows_alloc), cfg.hidden, cfg.num_topk
    mk = torch.zeros if zero else torch.empty
    out = {}
    if cfg.use_fp8:
        out["recv_x"] = mk((rows, H), dtype=torch.uint8, device="cuda")
        out["recv_sf"] = mk((int(info.sf_numel),), dtype=torch.float32, device="cuda")
    else:
        out["recv_x"] = mk((rows, H), dtype=torch.bfloat16, device="cuda")
        out["recv_sf"] = None
    if with_weights:
        shape = (rows,) if cfg.do_expand else (rows, K)
        out["recv_topk_weights"] = mk(shape, dtype=torch.float32, device="cuda")
    else:
        out["recv_topk_weights"] = None
    if with_idx and not cfg.do_expand:
        out["recv_topk_idx"] = mk((rows, K), dtype=torch.int32, device="cuda")
    else:
        out["recv_topk_idx"] = None
    return out


def alloc_recv(handle: Handle, with_weights: bool = False, with_idx: bool = False,
               zero: bool = False) -> dict:
    """Allocate the dispatch outputs for ``handle`` with torch (device memory only)."""
    return _alloc(handle.cfg, handle.info, with_weights, with_idx, zero)


def plan_layout(cfg: EpConfigC) -> EpLayoutInfoC:
    """Sizes of a do_cpu_sync = 0 layout (ep_plan_layout), before any GPU work."""
    info = EpLayoutInfoC()
    st = load_library().ep_plan_layout(ctypes.byref(cfg), ctypes.byref(info))
    if st != EP_OK:
        raise EpError(st, "ep_plan_layout")
    return info


def alloc_recv_planned(cfg: EpConfigC, with_weights: bool = False, with_idx: bool = False,
                       zero: bool = False) -> dict:
    """Allocate the dispatch outputs of a do_cpu_sync = 0 configuration from its plan."""
    return _alloc(cfg, plan_layout(cfg), with_weights, with_idx, zero)


def ep_layout_dispatch(cfg: EpConfigC, topk_idx: torch.Tensor, x: torch.Tensor,
                       topk_weights: Optional[torch.Tensor], recv_x: torch.Tensor,
                       recv_sf: Optional[torch.Tensor] = None,
                       recv_topk_weights: Optional[torch.Tensor] = None,
                       recv_topk_idx: Optional[torch.Tensor] = None, stream=None) -> Handle:
    """Layout and dispatch in one call (ep_layout_dispatch); returns the handle."""
    lib = load_library()
    if topk_idx.dtype not in (torch.int64, torch.int32):
        raise ValueError("topk_idx must be int64 or int32")
    if tuple(topk_idx.shape) != (cfg.num_tokens, cfg.num_topk):
        raise ValueError(f"topk_idx shape {tuple(topk_idx.shape)} != "
                         f"({cfg.num_tokens}, {cfg.num_topk})")
    if tuple(x.shape) != (cfg.num_tokens, cfg.hidden):
        raise ValueError(f"x shape {tuple(x.shape)} != ({cfg.num_tokens}, {cfg.hidden})")
    cfg.topk_idx_is_int64 = 1 if topk_idx.dtype == torch.int64 else 0
    h = ctypes.c_void_p(0)
    info = EpLayoutInfoC()
    st = lib.ep_layout_dispatch(
        ctypes.byref(cfg), _ptr(topk_idx, "topk_idx"), _ptr(x, "x", torch.bfloat16),
        _ptr(topk_weights, "topk_weights", torch.float32),
        _ptr(recv_x, "recv_x", (torch.bfloat16, torch.uint8, torch.float8_e4m3fn)),
        _ptr(recv_sf, "recv_sf", torch.float32),
        _ptr(recv_topk_weights, "recv_topk_weights", torch.float32),
        _ptr(recv_topk_idx, "recv_topk_idx", torch.int32), _stream_ptr(stream),
        ctypes.byref(h), ctypes.byref(info))
    if st != EP_OK:
        raise EpError(st, "ep_layout_dispatch")
    return Handle(h.value, EpConfigC.from_buffer_copy(cfg), info, st)


def ep_dispatch(handle: Handle, x: torch.Tensor, topk_weights: Optional[torch.Tensor],
                recv_x: torch.Tensor, recv_sf: Optional[torch.Tensor] = None,
                recv_topk_weights: Optional[torch.Tensor] = None,
                recv_topk_idx: Optional[torch.Tensor] = None, stream=None) -> None:
    lib = load_library()
    if tuple(x.shape) != (handle.T, handle.H):
        raise ValueError(f"x shape {tuple(x.shape)} != ({handle.T}, {handle.H})")
    st = lib.ep_dispatch(
        ctypes.c_void_p(handle.ptr), _ptr(x, "x", torch.bfloat16),
        _ptr(topk_weights, "topk_weights", torch.float32),
        _ptr(recv_x, "recv_x", (torch.bfloat16, torch.uint8, torch.float8_e4m3fn)),
        _ptr(recv_sf, "recv_sf", torch.float32),
        _ptr(recv_topk_weights, "recv_topk_weights", torch.float32),
        _ptr(recv_topk_idx, "recv_topk_idx", torch.int32), _stream_ptr(stream))
    if st != EP_OK:
        raise EpError(st, "ep_dispatch")


def ep_dispatch_fp8(handle: Handle, x_fp8: torch.Tensor, x_sf: torch.Tensor,
                    topk_weights: Optional[torch.Tensor], recv_x: torch.Tensor,
                    recv_sf: torch.Tensor, recv_topk_weights: Optional[torch.Tensor] = None,
                    recv_topk_idx: Optional[torch.Tensor] = None, stream=None) -> None:
    """Dispatch of a pre-quantised input: ``x_fp8`` e4m3 [T, H] (uint8 or
    float8_e4m3fn) and ``x_sf`` fp32 [T, H/128] with any non-negative strides
    (row-major, or a column-major view), copied without re-quantisation."""
    lib = load_library()
    if tuple(x_fp8.shape) != (handle.T, handle.H):
        raise ValueError(f"x_fp8 shape {tuple(x_fp8.shape)} != ({handle.T}, {handle.H})")
    if tuple(x_sf.shape) != (handle.T, handle.H // 128):
        raise ValueError(f"x_sf shape {tuple(x_sf.shape)} != ({handle.T}, {handle.H // 128})")
    if not x_sf.is_cuda or x_sf.dtype != torch.float32:
        raise ValueError("x_sf must be a CUDA float32 tensor")
    ts, hs = x_sf.stride()
    st = lib.ep_dispatch_fp8(
        ctypes.c_void_p(handle.ptr), _ptr(x_fp8, "x_fp8", (torch.uint8, torch.float8_e4m3fn)),
        x_sf.data_ptr() if x_sf.numel() > 0 else None, ts, hs,
        _ptr(topk_weights, "topk_weights", torch.float32),
        _ptr(recv_x, "recv_x", (torch.uint8, torch.float8_e4m3fn)),
        _ptr(recv_sf, "recv_sf", torch.float32),
        _ptr(recv_topk_weights, "recv_topk_weights", torch.float32),
        _ptr(recv_topk_idx, "recv_topk_idx", torch.int32), _stream_ptr(stream))
    if st != EP_OK:
        raise EpError(st, "ep_dispatch_fp8")


def ep_combine(handle: Handle, y: torch.Tensor, topk_weights: Optional[torch.Tensor] = None,
               bias_0: Optional[torch.Tensor] = None, bias_1: Optional[torch.Tensor] = None,
               expert_bias: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
               stream=None) -> torch.Tensor:
    lib = load_library()
    if y.dtype != torch.bfloat16:
        raise ValueError(f"combine requires bfloat16 expert output, got {y.dtype}")
    if out is None:
        out = torch.empty((handle.T, handle.H), dtype=torch.bfloat16, device=y.device)
    st = lib.ep_combine(
        ctypes.c_void_p(handle.ptr), _ptr(y, "y", torch.bfloat16),
        _ptr(topk_weights, "topk_weights", torch.float32), _ptr(bias_0, "bias_0", torch.bfloat16),
        _ptr(bias_1, "bias_1", torch.bfloat16), _ptr(expert_bias, "expert_bias", torch.bfloat16),
        _ptr(out, "out", torch.bfloat16), _stream_ptr(stream))
    if st != EP_OK:
        raise EpError(st, "ep_combine")
    return out


def ep_dispatch_backward(handle: Handle, grad_recv_x: torch.Tensor,
                         grad_recv_topk_weights: Optional[torch.Tensor] = None,
                         grad_x: Optional[torch.Tensor] = None,
                         grad_topk_weights: Optional[torch.Tensor] = None, stream=None):
    """Backward of dispatch: returns (grad_x [T, H] BF16, grad_topk_weights
    [T, K] fp32 or None)."""
    lib = load_library()
    if grad_recv_x.dtype != torch.bfloat16:
        raise ValueError(f"grad_recv_x must be bfloat16, got {grad_recv_x.dtype}")
    dev = grad_recv_x.device
    if grad_x is None:
        grad_x = torch.empty((handle.T, handle.H), dtype=torch.bfloat16, device=dev)
    if grad_recv_topk_weights is not None and grad_topk_weights is None:
        grad_topk_weights = torch.empty((handle.T, handle.K), dtype=torch.float32, device=dev)
    st = lib.ep_dispatch_backward(
        ctypes.c_void_p(handle.ptr), _ptr(grad_recv_x, "grad_recv_x", torch.bfloat16),
        _ptr(grad_recv_topk_weights, "grad_recv_topk_weights", torch.float32),
        _ptr(grad_x, "grad_x", torch.bfloat16),
        _ptr(grad_topk_weights, "grad_topk_weights", torch.float32), _stream_ptr(stream))
    if st != EP_OK:
        raise EpError(st, "ep_dispatch_backward")
    return grad_x, grad_topk_weights


def ep_combine_backward(handle: Handle, grad_combined_x: torch.Tensor,
                        grad_recv_x: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Backward of an unweighted combine: the BF16 gradient dispatched along
    the handle, [rows_alloc, H]."""
    lib = load_library()
    if tuple(grad_combined_x.shape) != (handle.T, handle.H):
        raise ValueError(f"grad shape {tuple(grad_combined_x.shape)} != ({handle.T}, {handle.H})")
    if grad_recv_x is None:
        grad_recv_x = torch.empty((handle.rows_alloc, handle.H), dtype=torch.bfloat16,
                                  device=grad_combined_x.device)
    st = lib.ep_combine_backward(
        ctypes.c_void_p(handle.ptr), _ptr(grad_combined_x, "grad_combined_x", torch.bfloat16),
        _ptr(grad_recv_x, "grad_recv_x", torch.bfloat16), _stream_ptr(stream))
    if st != EP_OK:
        raise EpError(st, "ep_combine_backward")
    return grad_recv_x


def ep_handle_free(handle: Handle) -> None:
    handle.free()


def host_wait_flag(flag: ctypes.c_int32, expected: int, timeout_ms: int) -> int:
    return load_library().ep_host_wait_flag(ctypes.byref(flag), expected, timeout_ms)


class EpLayoutBuffersC(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "topk_idx32", "cnt_expert", "cnt_expert_aligned", "psum_expert", "psum_padding",
        "cnt_rank", "psum_rank", "psum_rank_src", "dst_buffer_slot_idx", "recv_src_metadata",
        "is_token_in_rank", "status")]


EP_NOALLOC_SCRATCH_WORDS = 512 * 1024


def alloc_layout_buffers(cfg: EpConfigC, device="cuda") -> dict:
    """torch-allocated output buffers for ep_layout_noalloc (allocated by the caller)."""
    T, K, E, R = cfg.num_tokens, cfg.num_topk, cfg.num_experts, cfg.num_ranks
    rows = upper_bound_rows(cfg)
    i32 = dict(dtype=torch.int32, device=device)
    return {
        "topk_idx32": torch.empty((T, K), **i32),
        "cnt_expert": torch.empty((E,), **i32),
        "cnt_expert_aligned": torch.empty((E,), **i32),
        "psum_expert": torch.empty((E + 1,), **i32),
        "psum_padding": torch.empty((E + 1,), **i32),
        "cnt_rank": torch.empty((R,), **i32),
        "psum_rank": torch.empty((R + 1,), **i32),
        "psum_rank_src": torch.empty((R, R + 1), **i32),
        "dst_buffer_slot_idx": torch.empty((T, K), **i32),
        "recv_src_metadata": torch.empty((rows, 2), **i32),
        "is_token_in_rank": torch.empty((T, R), dtype=torch.uint8, device=device),
        "status": torch.empty((4,), **i32),
    }


def ep_layout_noalloc(cfg: EpConfigC, topk_idx: torch.Tensor, buffers: dict, stream=None) -> int:
    """Allocation-free layout into caller buffers; returns the ep_status code."""
    lib = load_library()
    fn = lib.ep_layout_noalloc
    fn.argtypes = [ctypes.POINTER(EpConfigC), ctypes.c_void_p, ctypes.POINTER(EpLayoutBuffersC),
                   ctypes.c_void_p]
    fn.restype = ctypes.c_int
    if topk_idx.dtype not in (torch.int64, torch.int32):
        raise ValueError("topk_idx must be int64 or int32")
    cfg.topk_idx_is_int64 = 1 if topk_idx.dtype == torch.int64 else 0
    b = EpLayoutBuffersC()
    for name, _ in EpLayoutBuffersC._fields_:
        t = buffers.get(name)
        setattr(b, name, None if t is None or t.numel() == 0 else t.data_ptr())
    p = topk_idx.data_ptr() if topk_idx.numel() > 0 else None
    return fn(ctypes.byref(cfg), p, ctypes.byref(b), _stream_ptr(stream))


def selftest_bounded_wait(wait_us: int, signal: bool, stream=None) -> int:
    """Runs the bounded-wait self-test; returns the EP_ERRBIT_* bits it reported."""
    lib = load_library()
    fn = lib.ep_selftest_bounded_wait
    fn.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(ctypes.c_uint32), ctypes.c_void_p]
    fn.restype = ctypes.c_int
    bits = ctypes.c_uint32(0xFFFFFFFF)
    st = fn(wait_us, 1 if signal else 0, ctypes.byref(bits), _stream_ptr(stream))
    if st != EP_OK:
        raise EpError(st, "ep_selftest_bounded_wait")
    return bits.value
