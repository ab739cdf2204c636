"""ctypes binding of ``libep_gb300.so`` -- the C ABI in ``include/ep.h``.

Argument marshalling only: every function takes torch tensors (or None for a
NULL pointer), checks dtype / device / contiguity, and passes raw device
pointers and the current CUDA stream to the library call of the same name.
All computation happens in the library's CUDA kernels; if the library is
missing this module raises instead of computing anything itself.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libep_gb300.so")

EP_OK, EP_ERR_INVALID_ARG, EP_ERR_CUDA, EP_ERR_CAPACITY, EP_ERR_BAD_EXPERT, EP_ERR_TIMEOUT, EP_ERR_STATE = range(7)
EP_BF16, EP_FP8_E4M3 = 0, 1
EP_LAYOUT_RANK_MAJOR, EP_LAYOUT_LOW_LATENCY, EP_LAYOUT_EXPERT_MAJOR = 0, 1, 2

_lock = threading.Lock()
_lib = None


class EPError(RuntimeError):
    def __init__(self, status: int, call: str):
        super().__init__(f"{call}: {status_str(status)} ({status})")
        self.status = status


def lib() -> ctypes.CDLL:
    """Load the CUDA library (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build the CUDA library first "
                    "(python -m combine_ep_get_03_gb300.build); there is no fallback path")
            L = ctypes.CDLL(LIB_PATH)
            P, I, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
            L.ep_handle_create.argtypes = [I, I, I, I, I, ctypes.POINTER(P)]
            L.ep_handle_destroy.argtypes = [P]
            L.ep_get_dispatch_layout.argtypes = [P, P, I, P, P, P, P]
            L.ep_get_num_recv.argtypes = [P, P, P, P, P]
            L.ep_dispatch.argtypes = [P, P, P, I, P, P, I64, P, P, P, I, P]
            L.ep_combine.argtypes = [P, P, I64, P, I, P]
            L.ep_combine_ex.argtypes = [P, I, P, P, I64, P, P, P, I, P]
            L.ep_handle_set_topk_idx_bits.argtypes = [P, I]
            L.ep_handle_topk_idx_bits.argtypes = [P]
            L.ep_handle_topk_idx_bits.restype = I
            L.ep_em_layout_and_dispatch.argtypes = [P, P, I, P, P, I, I, P, P, I64, I64, P, P, I, P]
            L.ep_em_dispatch.argtypes = [P, P, P, I, P, P, I64, I64, P, P, I, P]
            L.ep_em_get_layout.argtypes = [P, P, P, P]
            L.ep_em_combine.argtypes = [P, P, I64, P, I, P]
            L.ep_get_buffer_size_hint.argtypes = [I, I, I, I, I, I, I, I, P, P]
            L.ep_layout_and_dispatch.argtypes = [P, P, I, P, P, I, P, P, I64, P, P, P, I, P]
            L.ep_low_latency_dispatch.argtypes = [P, P, P, I, I, P, P, P, P, I, P]
            L.ep_low_latency_combine.argtypes = [P, P, P, P, I, P]
            L.ep_get_device_status.argtypes = [P, P]
            L.ep_check_wait_timeout.argtypes = [P, P]
            L.ep_get_dispatch_layout_noalloc.argtypes = [I, I, I, P, I, P, P, P, P, P, P, P, P, P, P]
            L.ep_status_str.argtypes = [I]
            L.ep_status_str.restype = ctypes.c_char_p
            for n in ("ep_handle_create", "ep_handle_destroy", "ep_get_dispatch_layout", "ep_get_num_recv",
                      "ep_dispatch", "ep_combine", "ep_layout_and_dispatch", "ep_low_latency_dispatch",
                      "ep_low_latency_combine", "ep_combine_ex", "ep_handle_set_topk_idx_bits",
                      "ep_em_layout_and_dispatch", "ep_em_dispatch", "ep_em_get_layout", "ep_em_combine",
                      "ep_get_buffer_size_hint",
                      "ep_get_device_status", "ep_check_wait_timeout", "ep_get_dispatch_layout_noalloc"):
                getattr(L, n).restype = I
            _lib = L
    return _lib


def status_str(s: int) -> str:
    return lib().ep_status_str(int(s)).decode()


ep_status_str = status_str


def _check(status: int, call: str) -> int:
    if status != EP_OK:
        raise EPError(status, call)
    return status


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream) -> int:
    if stream is None:
        # the current stream's handle without building a Stream object (a few
        # microseconds a call, which the low-latency calls notice)
        if _raw_stream is not None:
            return _raw_stream(torch.cuda.current_device())
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t, dtypes=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor or None")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtypes is not None and t.dtype not in dtypes:
        raise ValueError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    return t.data_ptr()


_FP8_BYTES = (torch.uint8, torch.float8_e4m3fn)


def _ids_ptr(h, topk_idx):
    """topk_idx must have the width the handle reads (int64 or int32)."""
    bits = lib().ep_handle_topk_idx_bits(h)
    return _ptr(topk_idx, (torch.int32,) if bits == 32 else (torch.int64,), "topk_idx")


# ------------------------------------------------------------------ calls

def ep_handle_create(num_ranks: int, num_experts: int, num_topk: int, hidden: int,
                     max_tokens_per_rank: int) -> int:
    h = ctypes.c_void_p()
    _check(lib().ep_handle_create(num_ranks, num_experts, num_topk, hidden, max_tokens_per_rank,
                                  ctypes.byref(h)), "ep_handle_create")
    return h.value


def ep_handle_set_topk_idx_bits(h: int, bits: int) -> None:
    _check(lib().ep_handle_set_topk_idx_bits(h, int(bits)), "ep_handle_set_topk_idx_bits")


def ep_handle_topk_idx_bits(h: int) -> int:
    return int(lib().ep_handle_topk_idx_bits(h))


def ep_handle_destroy(h: int) -> None:
    _check(lib().ep_handle_destroy(h), "ep_handle_destroy")


def ep_get_dispatch_layout(h, topk_idx, num_tokens_per_rank=None, num_tokens_per_expert=None,
                           is_token_in_rank=None, stream=None) -> None:
    T = topk_idx.shape[0]
    _check(lib().ep_get_dispatch_layout(
        h, _ids_ptr(h, topk_idx), T,
        _ptr(num_tokens_per_rank, (torch.int32,), "num_tokens_per_rank"),
        _ptr(num_tokens_per_expert, (torch.int32,), "num_tokens_per_expert"),
        _ptr(is_token_in_rank, (torch.bool, torch.uint8), "is_token_in_rank"),
        _stream(stream)), "ep_get_dispatch_layout")


def ep_get_num_recv(h, num_ranks: int, num_experts: int, stream=None, check: bool = True):
    """-> (num_recv_tokens_per_rank [R], num_recv_tokens_per_expert [E],
    rank_offset [R+1]) as numpy int32, plus the latched device status."""
    a = np.zeros(num_ranks, np.int32)
    b = np.zeros(num_experts, np.int32)
    c = np.zeros(num_ranks + 1, np.int32)
    st = lib().ep_get_num_recv(h, a.ctypes.data, b.ctypes.data, c.ctypes.data, _stream(stream))
    if check:
        _check(st, "ep_get_num_recv")
    return a, b, c, st


def ep_dispatch(h, x, topk_weights, dtype: int, recv_x, recv_scales=None, recv_src_idx=None,
                recv_topk_idx=None, recv_topk_weights=None, num_sms: int = 0, stream=None) -> None:
    fp8 = dtype == EP_FP8_E4M3
    cap = recv_x.shape[0] if recv_x is not None else 0
    _check(lib().ep_dispatch(
        h, _ptr(x, (torch.bfloat16,), "x"), _ptr(topk_weights, (torch.float32,), "topk_weights"), int(dtype),
        _ptr(recv_x, _FP8_BYTES if fp8 else (torch.bfloat16,), "recv_x"),
        _ptr(recv_scales, (torch.float32,), "recv_scales") if fp8 else None, cap,
        _ptr(recv_src_idx, (torch.int32,), "recv_src_idx"),
        _ptr(recv_topk_idx, (torch.int32,), "recv_topk_idx"),
        _ptr(recv_topk_weights, (torch.float32,), "recv_topk_weights"),
        int(num_sms), _stream(stream)), "ep_dispatch")


def ep_layout_and_dispatch(h, topk_idx, x, topk_weights, dtype: int, recv_x, recv_scales=None, recv_src_idx=None,
                           recv_topk_idx=None, recv_topk_weights=None, num_sms: int = 0, stream=None) -> None:
    fp8 = dtype == EP_FP8_E4M3
    cap = recv_x.shape[0] if recv_x is not None else 0
    _check(lib().ep_layout_and_dispatch(
        h, _ids_ptr(h, topk_idx), topk_idx.shape[0], _ptr(x, (torch.bfloat16,), "x"),
        _ptr(topk_weights, (torch.float32,), "topk_weights"), int(dtype),
        _ptr(recv_x, _FP8_BYTES if fp8 else (torch.bfloat16,), "recv_x"),
        _ptr(recv_scales, (torch.float32,), "recv_scales") if fp8 else None, cap,
        _ptr(recv_src_idx, (torch.int32,), "recv_src_idx"),
        _ptr(recv_topk_idx, (torch.int32,), "recv_topk_idx"),
        _ptr(recv_topk_weights, (torch.float32,), "recv_topk_weights"),
        int(num_sms), _stream(stream)), "ep_layout_and_dispatch")


def ep_combine(h, y, out, num_sms: int = 0, stream=None) -> None:
    _check(lib().ep_combine(h, _ptr(y, (torch.bfloat16,), "y"), y.shape[0],
                            _ptr(out, (torch.bfloat16,), "out"), int(num_sms), _stream(stream)), "ep_combine")


def ep_combine_ex(h, y, out, y_scales=None, recv_topk_weights=None, combined_topk_weights=None, num_sms: int = 0,
                  stream=None) -> None:
    """y bf16 [rows, H], or e4m3 bytes [rows, H] with fp32 y_scales [rows, H/128]."""
    fp8 = y_scales is not None
    _check(lib().ep_combine_ex(
        h, EP_FP8_E4M3 if fp8 else EP_BF16, _ptr(y, _FP8_BYTES if fp8 else (torch.bfloat16,), "y"),
        _ptr(y_scales, (torch.float32,), "y_scales"), y.shape[0],
        _ptr(recv_topk_weights, (torch.float32,), "recv_topk_weights"), _ptr(out, (torch.bfloat16,), "out"),
        _ptr(combined_topk_weights, (torch.float32,), "combined_topk_weights"), int(num_sms), _stream(stream)),
        "ep_combine_ex")


def ep_low_latency_dispatch(h, x, topk_idx, dtype: int, recv_x, recv_scales=None, recv_src_info=None,
                            recv_count=None, num_sms: int = 0, stream=None) -> None:
    fp8 = dtype == EP_FP8_E4M3
    _check(lib().ep_low_latency_dispatch(
        h, _ptr(x, (torch.bfloat16,), "x"), _ids_ptr(h, topk_idx), topk_idx.shape[0],
        int(dtype), _ptr(recv_x, _FP8_BYTES if fp8 else (torch.bfloat16,), "recv_x"),
        _ptr(recv_scales, (torch.float32,), "recv_scales") if fp8 else None,
        _ptr(recv_src_info, (torch.int32,), "recv_src_info"), _ptr(recv_count, (torch.int32,), "recv_count"),
        int(num_sms), _stream(stream)), "ep_low_latency_dispatch")


def ep_low_latency_combine(h, y, topk_weights, out, num_sms: int = 0, stream=None) -> None:
    _check(lib().ep_low_latency_combine(
        h, _ptr(y, (torch.bfloat16,), "y"), _ptr(topk_weights, (torch.float32,), "topk_weights"),
        _ptr(out, (torch.bfloat16,), "out"), int(num_sms), _stream(stream)), "ep_low_latency_combine")


def _em_out(h, dtype, topk_weights, recv_x, recv_scales, recv_src_idx, recv_weights):
    fp8 = dtype == EP_FP8_E4M3
    cap = recv_x.shape[0] if recv_x is not None else 0
    if fp8 and recv_scales is not None and (recv_scales.dim() != 2 or recv_scales.stride(1) != 1):
        raise ValueError("recv_scales must be a contiguous [H/128, scales_ld] tensor")
    ld = recv_scales.shape[1] if (fp8 and recv_scales is not None) else 0
    return (_ptr(topk_weights, (torch.float32,), "topk_weights"), int(dtype),
            _ptr(recv_x, _FP8_BYTES if fp8 else (torch.bfloat16,), "recv_x"),
            _ptr(recv_scales, (torch.float32,), "recv_scales") if fp8 else None, ld, cap,
            _ptr(recv_src_idx, (torch.int32,), "recv_src_idx"), _ptr(recv_weights, (torch.float32,), "recv_weights"))


def ep_em_layout_and_dispatch(h, topk_idx, x, topk_weights, dtype: int, expert_alignment: int, recv_x,
                              recv_scales=None, recv_src_idx=None, recv_weights=None, num_sms: int = 0,
                              stream=None) -> None:
    w, dt, rx, rs, ld, cap, si, rw = _em_out(h, dtype, topk_weights, recv_x, recv_scales, recv_src_idx, recv_weights)
    _check(lib().ep_em_layout_and_dispatch(h, _ids_ptr(h, topk_idx), topk_idx.shape[0],
                                           _ptr(x, (torch.bfloat16,), "x"), w, dt, int(expert_alignment), rx, rs,
                                           ld, cap, si, rw, int(num_sms), _stream(stream)),
           "ep_em_layout_and_dispatch")


def ep_em_dispatch(h, x, topk_weights, dtype: int, recv_x, recv_scales=None, recv_src_idx=None, recv_weights=None,
                   num_sms: int = 0, stream=None) -> None:
    w, dt, rx, rs, ld, cap, si, rw = _em_out(h, dtype, topk_weights, recv_x, recv_scales, recv_src_idx, recv_weights)
    _check(lib().ep_em_dispatch(h, _ptr(x, (torch.bfloat16,), "x"), w, dt, rx, rs, ld, cap, si, rw, int(num_sms),
                                _stream(stream)), "ep_em_dispatch")


def ep_em_get_layout(h, num_experts: int, stream=None, check: bool = True):
    """-> (num_recv_tokens_per_expert [E], expert_offset [E+1]) numpy int32, status."""
    a = np.zeros(num_experts, np.int32)
    b = np.zeros(num_experts + 1, np.int32)
    st = lib().ep_em_get_layout(h, a.ctypes.data, b.ctypes.data, _stream(stream))
    if check:
        _check(st, "ep_em_get_layout")
    return a, b, st


def ep_em_combine(h, y, out, num_sms: int = 0, stream=None) -> None:
    _check(lib().ep_em_combine(h, _ptr(y, (torch.bfloat16,), "y"), y.shape[0], _ptr(out, (torch.bfloat16,), "out"),
                               int(num_sms), _stream(stream)), "ep_em_combine")


def ep_get_buffer_size_hint(num_ranks, num_experts, num_topk, hidden, max_tokens_per_rank, dtype: int,
                            layout: int, expert_alignment: int = 1):
    """-> (rows, bytes): the largest receive buffers any routing can need."""
    rows, nbytes = ctypes.c_int64(), ctypes.c_int64()
    _check(lib().ep_get_buffer_size_hint(num_ranks, num_experts, num_topk, hidden, max_tokens_per_rank, int(dtype),
                                         int(layout), int(expert_alignment), ctypes.byref(rows),
                                         ctypes.byref(nbytes)), "ep_get_buffer_size_hint")
    return rows.value, nbytes.value


def ep_get_device_status(h, stream=None) -> int:
    """Synchronise, then return and clear the latched device status."""
    return lib().ep_get_device_status(h, _stream(stream))


def ep_check_wait_timeout(h, stream=None) -> None:
    """Enqueue the bounded-wait self-check (waits that cannot complete give
    up and latch EP_ERR_TIMEOUT; read it with ep_get_device_status)."""
    _check(lib().ep_check_wait_timeout(h, _stream(stream)), "ep_check_wait_timeout")


def ep_get_dispatch_layout_noalloc(num_ranks, num_experts, num_topk, topk_idx, num_recv_tokens_per_rank,
                                   num_recv_tokens_per_expert, rank_offset, token_dest, topk_idx32,
                                   num_tokens_per_rank=None, num_tokens_per_expert=None, is_token_in_rank=None,
                                   device_status=None, stream=None) -> None:
    """The handle-free, allocation-free layout: every output is a caller tensor
    (see include/ep.h for shapes); the scan state lives in the library."""
    R, E, k = num_ranks, num_experts, num_topk
    if not isinstance(topk_idx, torch.Tensor) or topk_idx.dim() != 2 or topk_idx.shape[1] != k:
        raise ValueError(f"topk_idx must be a [T, {k}] tensor (num_topk columns)")
    T = topk_idx.shape[0]
    kmax = min(k, R)
    for t, n, name in ((num_recv_tokens_per_rank, R, "num_recv_tokens_per_rank"),
                       (num_recv_tokens_per_expert, E, "num_recv_tokens_per_expert"),
                       (rank_offset, R + 1, "rank_offset"), (token_dest, T * kmax * 2, "token_dest"),
                       (topk_idx32, T * k, "topk_idx32"), (num_tokens_per_rank, R * R, "num_tokens_per_rank"),
                       (num_tokens_per_expert, R * E, "num_tokens_per_expert"),
                       (is_token_in_rank, T * R, "is_token_in_rank"), (device_status, 1, "device_status")):
        if t is not None and t.numel() < n:
            raise ValueError(f"{name} holds {t.numel()} elements, the call needs {n}")
    _check(lib().ep_get_dispatch_layout_noalloc(
        R, E, k, _ptr(topk_idx, (torch.int64,), "topk_idx"), T,
        _ptr(num_tokens_per_rank, (torch.int32,), "num_tokens_per_rank"),
        _ptr(num_tokens_per_expert, (torch.int32,), "num_tokens_per_expert"),
        _ptr(is_token_in_rank, (torch.bool, torch.uint8), "is_token_in_rank"),
        _ptr(num_recv_tokens_per_rank, (torch.int32,), "num_recv_tokens_per_rank"),
        _ptr(num_recv_tokens_per_expert, (torch.int32,), "num_recv_tokens_per_expert"),
        _ptr(rank_offset, (torch.int32,), "rank_offset"), _ptr(token_dest, (torch.int32,), "token_dest"),
        _ptr(topk_idx32, (torch.int32,), "topk_idx32"), _ptr(device_status, (torch.int32,), "device_status"),
        _stream(stream)), "ep_get_dispatch_layout_noalloc")


class Handle:
    """Owns one ep_handle_t; methods call the ABI functions of the same name
    after checking that every buffer is large enough for the call."""

    def __init__(self, num_ranks, num_experts, num_topk, hidden, max_tokens_per_rank):
        self.R, self.E, self.k, self.H = num_ranks, num_experts, num_topk, hidden
        self.max_tokens_per_rank = max_tokens_per_rank
        self.T = None      # tokens of the last layout
        self.T_ll = None   # tokens of the last low-latency dispatch
        self.T_em = None   # tokens of the last expert-major layout
        self.ptr = ep_handle_create(num_ranks, num_experts, num_topk, hidden, max_tokens_per_rank)

    @property
    def topk_idx_bits(self) -> int:
        return ep_handle_topk_idx_bits(self.ptr)

    def set_topk_idx_bits(self, bits: int) -> None:
        ep_handle_set_topk_idx_bits(self.ptr, bits)

    @property
    def M(self) -> int:
        """Rows per expert in the low-latency receive buffer."""
        return self.R * self.max_tokens_per_rank

    @property
    def G(self) -> int:
        return self.H // 128

    def close(self):
        if getattr(self, "ptr", None):
            ep_handle_destroy(self.ptr)
            self.ptr = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    @staticmethod
    def _need(t, n, name):
        if t is not None and t.numel() < n:
            raise ValueError(f"{name} holds {t.numel()} elements, the call needs {n}")

    def get_dispatch_layout(self, topk_idx, num_tokens_per_rank=None, num_tokens_per_expert=None,
                            is_token_in_rank=None, stream=None):
        T = topk_idx.shape[0]
        if topk_idx.dim() != 2 or topk_idx.shape[1] != self.k:
            raise ValueError(f"topk_idx must be [T, {self.k}]")
        self._need(num_tokens_per_rank, self.R * self.R, "num_tokens_per_rank")
        self._need(num_tokens_per_expert, self.R * self.E, "num_tokens_per_expert")
        self._need(is_token_in_rank, T * self.R, "is_token_in_rank")
        ep_get_dispatch_layout(self.ptr, topk_idx, num_tokens_per_rank, num_tokens_per_expert,
                               is_token_in_rank, stream)
        self.T = T

    def get_num_recv(self, stream=None, check=True):
        return ep_get_num_recv(self.ptr, self.R, self.E, stream=stream, check=check)

    def dispatch(self, x, topk_weights, dtype, recv_x, recv_scales=None, recv_src_idx=None,
                 recv_topk_idx=None, recv_topk_weights=None, num_sms=0, stream=None):
        if self.T is None:
            raise RuntimeError("dispatch before any layout on this handle")
        cap = recv_x.shape[0]
        if recv_x.dim() != 2 or recv_x.shape[1] != self.H:
            raise ValueError(f"recv_x must be [cap, {self.H}]")
        self._need(x, self.T * self.H, "x")
        self._need(topk_weights, self.T * self.k, "topk_weights")
        if dtype == EP_FP8_E4M3:
            if recv_scales is None:
                raise ValueError("FP8 dispatch needs recv_scales")
            self._need(recv_scales, cap * self.G, "recv_scales")
        self._need(recv_src_idx, cap, "recv_src_idx")
        self._need(recv_topk_idx, cap * self.k, "recv_topk_idx")
        self._need(recv_topk_weights, cap * self.k, "recv_topk_weights")
        ep_dispatch(self.ptr, x, topk_weights, dtype, recv_x, recv_scales, recv_src_idx, recv_topk_idx,
                    recv_topk_weights, num_sms, stream)

    def layout_and_dispatch(self, topk_idx, x, topk_weights, dtype, recv_x, recv_scales=None, recv_src_idx=None,
                            recv_topk_idx=None, recv_topk_weights=None, num_sms=0, stream=None):
        T = topk_idx.shape[0]
        if topk_idx.dim() != 2 or topk_idx.shape[1] != self.k:
            raise ValueError(f"topk_idx must be [T, {self.k}]")
        cap = recv_x.shape[0]
        if recv_x.dim() != 2 or recv_x.shape[1] != self.H:
            raise ValueError(f"recv_x must be [cap, {self.H}]")
        self._need(x, T * self.H, "x")
        self._need(topk_weights, T * self.k, "topk_weights")
        if dtype == EP_FP8_E4M3:
            if recv_scales is None:
                raise ValueError("FP8 dispatch needs recv_scales")
            self._need(recv_scales, cap * self.G, "recv_scales")
        self._need(recv_src_idx, cap, "recv_src_idx")
        self._need(recv_topk_idx, cap * self.k, "recv_topk_idx")
        self._need(recv_topk_weights, cap * self.k, "recv_topk_weights")
        ep_layout_and_dispatch(self.ptr, topk_idx, x, topk_weights, dtype, recv_x, recv_scales, recv_src_idx,
                               recv_topk_idx, recv_topk_weights, num_sms, stream)
        self.T = T

    def combine(self, y, out, num_sms=0, stream=None):
        if self.T is None:
            raise RuntimeError("combine before any layout on this handle")
        if y.dim() != 2 or y.shape[1] != self.H:
            raise ValueError(f"y must be [rows, {self.H}]")
        self._need(out, self.T * self.H, "out")
        ep_combine(self.ptr, y, out, num_sms, stream)

    def combine_ex(self, y, out, y_scales=None, recv_topk_weights=None, combined_topk_weights=None, num_sms=0,
                   stream=None):
        if self.T is None:
            raise RuntimeError("combine before any layout on this handle")
        if y.dim() != 2 or y.shape[1] != self.H:
            raise ValueError(f"y must be [rows, {self.H}]")
        rows = y.shape[0]
        self._need(out, self.T * self.H, "out")
        self._need(y_scales, rows * self.G, "y_scales")
        self._need(recv_topk_weights, rows * self.k, "recv_topk_weights")
        self._need(combined_topk_weights, self.T * self.k, "combined_topk_weights")
        ep_combine_ex(self.ptr, y, out, y_scales, recv_topk_weights, combined_topk_weights, num_sms, stream)

    def low_latency_dispatch(self, x, topk_idx, dtype, recv_x, recv_scales=None, recv_src_info=None,
                             recv_count=None, num_sms=0, stream=None):
        T = topk_idx.shape[0]
        if topk_idx.dim() != 2 or topk_idx.shape[1] != self.k:
            raise ValueError(f"topk_idx must be [T, {self.k}]")
        rows = self.E * self.M
        self._need(x, T * self.H, "x")
        if recv_x.numel() < rows * self.H:
            raise ValueError(f"recv_x must hold [E, M, H] = [{self.E}, {self.M}, {self.H}]")
        if dtype == EP_FP8_E4M3:
            if recv_scales is None:
                raise ValueError("FP8 dispatch needs recv_scales")
            self._need(recv_scales, rows * self.G, "recv_scales")
        self._need(recv_src_info, rows, "recv_src_info")
        self._need(recv_count, self.E, "recv_count")
        ep_low_latency_dispatch(self.ptr, x, topk_idx, dtype, recv_x, recv_scales, recv_src_info, recv_count,
                                num_sms, stream)
        self.T_ll = T

    def low_latency_combine(self, y, topk_weights, out, num_sms=0, stream=None):
        if self.T_ll is None:
            raise RuntimeError("low-latency combine before any low-latency dispatch")
        if y.numel() < self.E * self.M * self.H:
            raise ValueError(f"y must hold [E, M, H] = [{self.E}, {self.M}, {self.H}]")
        self._need(topk_weights, self.T_ll * self.k, "topk_weights")
        self._need(out, self.T_ll * self.H, "out")
        ep_low_latency_combine(self.ptr, y, topk_weights, out, num_sms, stream)

    # -------------------------------------------------------- expert-major

    def _em_need(self, T, topk_weights, dtype, recv_x, recv_scales, recv_src_idx, recv_weights):
        if recv_x.dim() != 2 or recv_x.shape[1] != self.H:
            raise ValueError(f"recv_x must be [cap, {self.H}]")
        cap = recv_x.shape[0]
        self._need(topk_weights, T * self.k, "topk_weights")
        if dtype == EP_FP8_E4M3:
            if recv_scales is None or recv_scales.dim() != 2 or recv_scales.shape[0] != self.G:
                raise ValueError(f"FP8 dispatch needs recv_scales [{self.G}, scales_ld]")
            if recv_scales.shape[1] < cap:
                raise ValueError("scales_ld must be >= the capacity rows")
        self._need(recv_src_idx, cap, "recv_src_idx")
        self._need(recv_weights, cap, "recv_weights")

    def em_layout_and_dispatch(self, topk_idx, x, topk_weights, dtype, expert_alignment, recv_x, recv_scales=None,
                               recv_src_idx=None, recv_weights=None, num_sms=0, stream=None):
        T = topk_idx.shape[0]
        if topk_idx.dim() != 2 or topk_idx.shape[1] != self.k:
            raise ValueError(f"topk_idx must be [T, {self.k}]")
        self._need(x, T * self.H, "x")
        self._em_need(T, topk_weights, dtype, recv_x, recv_scales, recv_src_idx, recv_weights)
        ep_em_layout_and_dispatch(self.ptr, topk_idx, x, topk_weights, dtype, expert_alignment, recv_x, recv_scales,
                                  recv_src_idx, recv_weights, num_sms, stream)
        self.T_em = T

    def em_dispatch(self, x, topk_weights, dtype, recv_x, recv_scales=None, recv_src_idx=None, recv_weights=None,
                    num_sms=0, stream=None):
        if self.T_em is None:
            raise RuntimeError("expert-major dispatch before any expert-major layout")
        self._need(x, self.T_em * self.H, "x")
        self._em_need(self.T_em, topk_weights, dtype, recv_x, recv_scales, recv_src_idx, recv_weights)
        ep_em_dispatch(self.ptr, x, topk_weights, dtype, recv_x, recv_scales, recv_src_idx, recv_weights, num_sms,
                       stream)

    def em_get_layout(self, stream=None, check=True):
        return ep_em_get_layout(self.ptr, self.E, stream=stream, check=check)

    def em_combine(self, y, out, num_sms=0, stream=None):
        if self.T_em is None:
            raise RuntimeError("expert-major combine before any expert-major layout")
        if y.dim() != 2 or y.shape[1] != self.H:
            raise ValueError(f"y must be [rows, {self.H}]")
        self._need(out, self.T_em * self.H, "out")
        ep_em_combine(self.ptr, y, out, num_sms, stream)

    def get_device_status(self, stream=None):
        return ep_get_device_status(self.ptr, stream)

    def check_wait_timeout(self, stream=None):
        ep_check_wait_timeout(self.ptr, stream)
