"""TEST INFRASTRUCTURE ONLY -- Python access to the CPU oracle.

The oracle (``ep_oracle.cpp``) is a plain, slow, single-threaded C++
statement of MoE expert-parallel dispatch / combine written from the pages
("DeepEP 要約" section 3; the vi.news.hada.io DeepEP article, section
"Mẫu sử dụng cho huấn luyện, prefill và decoding").  Only the tests, the
package smoke check and the benchmark's CPU-baseline leg may import this
module; the product path never does.  It shares no code with the CUDA
library.

Arrays are numpy; bf16 tensors travel as uint16 bit patterns.  The
row-moving steps take ``threads=n`` to run the same definitions with their
token loop split over n host threads (``ep_oracle_threads.cpp``; results are
byte-identical), which only the CPU-baseline timing uses.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ep_oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "libep_oracle.so")
_SRC_THREADS = os.path.join(_HERE, "ep_oracle_threads.cpp")
_LIB_THREADS = os.path.join(_HERE, "libep_oracle_threads.so")
_lock = threading.Lock()
_lib = None
_lib_threads = None

OK, INVALID_ARG, CAPACITY, BAD_EXPERT = 0, 1, 3, 4


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (contraction off: one IEEE op per + and *)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "ep_oracle.h"))
    ):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-o", tmp, _SRC]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    build_threads(force)
    return _LIB_PATH


def build_threads(force: bool = False) -> str:
    """Compile the multi-threaded copy (ep_oracle_threads.cpp, which includes
    the oracle's own source and splits its token loops over std::threads)."""
    deps = [_SRC, os.path.join(_HERE, "ep_oracle.h"), _SRC_THREADS]
    if force or not os.path.exists(_LIB_THREADS) or os.path.getmtime(_LIB_THREADS) < max(
        os.path.getmtime(d) for d in deps
    ):
        tmp = _LIB_THREADS + f".tmp{os.getpid()}"
        cmd = ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-pthread",
               "-shared", "-o", tmp, _SRC_THREADS]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_THREADS)
    return _LIB_THREADS


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            I64 = ctypes.c_int64
            lib.ref_float_to_e4m3.argtypes = [ctypes.c_float]
            lib.ref_float_to_e4m3.restype = ctypes.c_uint8
            lib.ref_e4m3_to_float.argtypes = [ctypes.c_uint8]
            lib.ref_e4m3_to_float.restype = ctypes.c_float
            lib.ref_float_to_bf16.argtypes = [ctypes.c_float]
            lib.ref_float_to_bf16.restype = ctypes.c_uint16
            lib.ref_quantize_row.argtypes = [I, P, P, P]
            lib.ref_layout.argtypes = [I, I, I, I, P, P, P, P, P, P, P, P]
            lib.ref_dispatch.argtypes = [I, I, I, I, I, I, P, P, P, I64, P, P, P, P, P]
            lib.ref_combine.argtypes = [I, I, I, I, I, P, P, I64, P]
            lib.ref_ll_dispatch.argtypes = [I, I, I, I, I, I, I, P, P, P, P, P, P, P]
            lib.ref_ll_combine.argtypes = [I, I, I, I, I, I, P, P, P, P]
            lib.ref_combine_ex.argtypes = [I, I, I, I, I, P, I, P, P, I64, P, P, P]
            lib.ref_em_layout.argtypes = [I, I, I, I, P, I, P, P, P]
            lib.ref_em_dispatch.argtypes = [I, I, I, I, I, I, P, P, P, I, I64, P, P, I64, P, P]
            lib.ref_em_combine.argtypes = [I, I, I, I, I, P, I, P, I64, P]
            for name in ("ref_quantize_row", "ref_layout", "ref_dispatch", "ref_combine",
                         "ref_ll_dispatch", "ref_ll_combine", "ref_combine_ex", "ref_em_layout",
                         "ref_em_dispatch", "ref_em_combine"):
                getattr(lib, name).restype = I
            _lib = lib
    return _lib


def _load_threads():
    global _lib_threads
    with _lock:
        if _lib_threads is None:
            lib = ctypes.CDLL(build_threads())
            P, I, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
            lib.ref_threads_available.argtypes = []
            lib.ref_threads_dispatch.argtypes = [I, I, I, I, I, I, I, P, P, P, I64, P, P, P, P, P]
            lib.ref_threads_combine.argtypes = [I, I, I, I, I, I, P, P, I64, P]
            lib.ref_threads_combine_ex.argtypes = [I, I, I, I, I, I, P, I, P, P, I64, P, P, P]
            lib.ref_threads_ll_dispatch.argtypes = [I, I, I, I, I, I, I, I, P, P, P, P, P, P, P]
            lib.ref_threads_ll_combine.argtypes = [I, I, I, I, I, I, I, P, P, P, P]
            for name in ("ref_threads_available", "ref_threads_dispatch", "ref_threads_combine",
                         "ref_threads_combine_ex", "ref_threads_ll_dispatch", "ref_threads_ll_combine"):
                getattr(lib, name).restype = I
            _lib_threads = lib
    return _lib_threads


def threads_available() -> int:
    """Host cores this process may run on (sched_getaffinity)."""
    return int(_load_threads().ref_threads_available())


def _step(name, threads):
    """The single-threaded oracle function, or (threads = n) its copy whose
    token loop runs on n threads -- byte-identical results."""
    if threads is None:
        return getattr(_load(), "ref_" + name)
    f = getattr(_load_threads(), "ref_threads_" + name)
    return lambda *a: f(int(threads), *a)


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    a = np.ascontiguousarray(a)
    assert a.dtype == dtype, (a.dtype, dtype)
    return a


class OracleError(RuntimeError):
    def __init__(self, status):
        super().__init__(f"oracle status {status}")
        self.status = status


def _check(st, allow=(OK,)):
    if st not in allow:
        raise OracleError(st)
    return st


# ----------------------------------------------------------------- formats

def float_to_e4m3(f: float) -> int:
    return int(_load().ref_float_to_e4m3(float(f)))


def e4m3_to_float(code: int) -> float:
    return float(_load().ref_e4m3_to_float(int(code)))


def float_to_bf16(f: float) -> int:
    return int(_load().ref_float_to_bf16(float(f)))


def float_to_e4m3_array(v: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.ascontiguousarray(v, dtype=np.float32).ravel()
    return np.fromiter((lib.ref_float_to_e4m3(float(x)) for x in flat), dtype=np.uint8,
                       count=flat.size).reshape(np.shape(v))


def quantize_row(x_bits: np.ndarray):
    """One bf16 row (uint16 [H]) -> (e4m3 bytes [H], fp32 scales [H/128])."""
    x_bits = _c(x_bits, np.uint16)
    H = x_bits.size
    q = np.zeros(H, np.uint8)
    s = np.zeros(max(H // 128, 1), np.float32)
    _check(_load().ref_quantize_row(H, _p(x_bits), _p(q), _p(s)))
    return q, s[: H // 128]


# ----------------------------------------------------------------- steps

def layout(R, E, k, topk_idx):
    """get_dispatch_layout; returns a dict of numpy arrays."""
    idx = _c(topk_idx, np.int64)
    T = idx.shape[0]
    out = dict(
        num_tokens_per_rank=np.zeros((R, R), np.int32),
        num_tokens_per_expert=np.zeros((R, E), np.int32),
        is_token_in_rank=np.zeros((T, R), np.uint8),   # 0/1 bytes, as written
        slot=np.zeros((T, R), np.int32),
        num_recv_per_rank=np.zeros(R, np.int32),
        rank_offset=np.zeros(R + 1, np.int32),
        num_recv_per_expert=np.zeros(E, np.int32),
    )
    _check(_load().ref_layout(R, E, k, T, _p(idx), *(_p(out[n]) for n in (
        "num_tokens_per_rank", "num_tokens_per_expert", "is_token_in_rank", "slot",
        "num_recv_per_rank", "rank_offset", "num_recv_per_expert"))))
    return out


def dispatch(R, E, k, x_bits, topk_idx, topk_weights, fp8, capacity_rows=None, threads=None):
    """Normal dispatch.  Returns (dict of outputs, status)."""
    x_bits = _c(x_bits, np.uint16)
    idx = _c(topk_idx, np.int64)
    T, H = x_bits.shape
    if capacity_rows is None:
        capacity_rows = int(layout(R, E, k, idx)["rank_offset"][-1])
    rows = max(int(capacity_rows), 1)
    w = None if topk_weights is None else _c(topk_weights, np.float32)
    out = dict(
        recv_x=np.zeros((rows, H), np.uint8 if fp8 else np.uint16),
        recv_scales=np.zeros((rows, H // 128), np.float32) if fp8 else None,
        recv_src_idx=np.full(rows, -7, np.int32),
        recv_topk_idx=np.full((rows, k), -7, np.int32),
        recv_topk_weights=np.full((rows, k), -7.0, np.float32),
    )
    st = _check(_step("dispatch", threads)(R, E, k, T, H, int(bool(fp8)), _p(x_bits), _p(idx), _p(w),
                                     int(capacity_rows), _p(out["recv_x"]), _p(out["recv_scales"]),
                                     _p(out["recv_src_idx"]), _p(out["recv_topk_idx"]),
                                     _p(out["recv_topk_weights"])), allow=(OK, CAPACITY))
    if capacity_rows == 0:
        for key in out:
            if out[key] is not None:
                out[key] = out[key][:0]
    return out, st


def combine(R, E, k, topk_idx, y_bits, threads=None):
    """Normal combine: y (uint16 [rows, H]) -> out (uint16 [T, H])."""
    idx = _c(topk_idx, np.int64)
    y_bits = _c(y_bits, np.uint16)
    T = idx.shape[0]
    H = y_bits.shape[1]
    out = np.zeros((T, H), np.uint16)
    _check(_step("combine", threads)(R, E, k, T, H, _p(idx), _p(y_bits), y_bits.shape[0], _p(out)))
    return out


def ll_dispatch(R, E, k, M, x_bits, topk_idx, fp8, threads=None):
    """Low-latency dispatch into [E, M, H].  Returns (dict, status)."""
    x_bits = _c(x_bits, np.uint16)
    idx = _c(topk_idx, np.int64)
    T, H = x_bits.shape
    out = dict(
        recv_x=np.zeros((E, M, H), np.uint8 if fp8 else np.uint16),
        recv_scales=np.zeros((E, M, H // 128), np.float32) if fp8 else None,
        recv_src_info=np.full((E, M), -7, np.int32),
        recv_count=np.zeros(E, np.int32),
        slot=np.zeros((T, k), np.int32),
    )
    st = _check(_step("ll_dispatch", threads)(R, E, k, T, H, M, int(bool(fp8)), _p(x_bits), _p(idx),
                                        _p(out["recv_x"]), _p(out["recv_scales"]),
                                        _p(out["recv_src_info"]), _p(out["recv_count"]),
                                        _p(out["slot"])), allow=(OK, CAPACITY))
    return out, st


def ll_combine(R, E, k, M, topk_idx, topk_weights, y_bits, threads=None):
    """Low-latency combine: y (uint16 [E, M, H]) -> out (uint16 [T, H])."""
    idx = _c(topk_idx, np.int64)
    w = _c(topk_weights, np.float32)
    y_bits = _c(y_bits, np.uint16)
    T = idx.shape[0]
    H = y_bits.shape[-1]
    out = np.zeros((T, H), np.uint16)
    _check(_step("ll_combine", threads)(R, E, k, T, H, M, _p(idx), _p(w), _p(y_bits), _p(out)))
    return out


def combine_ex(R, E, k, topk_idx, y, y_scales=None, recv_topk_weights=None, threads=None):
    """Normal combine, general form.  y is uint16 bf16 bits [rows, H], or
    uint8 e4m3 bytes [rows, H] with fp32 y_scales [rows, H/128].  With
    recv_topk_weights [rows, k] the weights are summed back too.  Returns
    (out uint16 [T, H], combined weights float32 [T, k] or None)."""
    idx = _c(topk_idx, np.int64)
    fp8 = y_scales is not None
    y = _c(y, np.uint8 if fp8 else np.uint16)
    sc = None if y_scales is None else _c(y_scales, np.float32)
    rw = None if recv_topk_weights is None else _c(recv_topk_weights, np.float32)
    T = idx.shape[0]
    H = y.shape[1]
    out = np.zeros((T, H), np.uint16)
    cw = None if rw is None else np.zeros((T, k), np.float32)
    _check(_step("combine_ex", threads)(R, E, k, T, H, _p(idx), int(fp8), _p(y), _p(sc), y.shape[0], _p(rw),
                                  _p(out), _p(cw)))
    return out, cw


def em_layout(R, E, k, topk_idx, align):
    """Expert-major layout: dict(num_recv_per_expert [E], expert_offset [E+1],
    row [T, k])."""
    idx = _c(topk_idx, np.int64)
    T = idx.shape[0]
    out = dict(num_recv_per_expert=np.zeros(E, np.int32), expert_offset=np.zeros(E + 1, np.int32),
               row=np.zeros((T, k), np.int32))
    _check(_load().ref_em_layout(R, E, k, T, _p(idx), int(align), _p(out["num_recv_per_expert"]),
                                 _p(out["expert_offset"]), _p(out["row"])))
    return out


def em_dispatch(R, E, k, x_bits, topk_idx, topk_weights, fp8, align, capacity_rows=None, scales_ld=None):
    """Expert-major dispatch.  Returns (dict, status); recv_scales is
    group-major [H/128, scales_ld]; rows the oracle does not write keep the
    fill values (recv_x 0, scales -7, src_idx -7, weights -7)."""
    x_bits = _c(x_bits, np.uint16)
    idx = _c(topk_idx, np.int64)
    T, H = x_bits.shape
    if capacity_rows is None:
        capacity_rows = int(em_layout(R, E, k, idx, align)["expert_offset"][-1])
    if scales_ld is None:
        scales_ld = (int(capacity_rows) + 3) // 4 * 4
    rows = max(int(capacity_rows), 1)
    w = None if topk_weights is None else _c(topk_weights, np.float32)
    out = dict(
        recv_x=np.zeros((rows, H), np.uint8 if fp8 else np.uint16),
        recv_scales=np.full((H // 128, max(scales_ld, 1)), -7.0, np.float32) if fp8 else None,
        recv_src_idx=np.full(rows, -7, np.int32),
        recv_weights=np.full(rows, -7.0, np.float32),
    )
    st = _check(_load().ref_em_dispatch(R, E, k, T, H, int(bool(fp8)), _p(x_bits), _p(idx), _p(w), int(align),
                                        int(capacity_rows), _p(out["recv_x"]), _p(out["recv_scales"]),
                                        int(scales_ld), _p(out["recv_src_idx"]), _p(out["recv_weights"])),
                allow=(OK, CAPACITY))
    if capacity_rows == 0:
        for key in ("recv_x", "recv_src_idx", "recv_weights"):
            out[key] = out[key][:0]
    return out, st


def em_combine(R, E, k, topk_idx, align, y_bits):
    """Expert-major combine: y (uint16 [rows, H]) -> out (uint16 [T, H])."""
    idx = _c(topk_idx, np.int64)
    y_bits = _c(y_bits, np.uint16)
    T = idx.shape[0]
    H = y_bits.shape[1]
    out = np.zeros((T, H), np.uint16)
    _check(_load().ref_em_combine(R, E, k, T, H, _p(idx), int(align), _p(y_bits), y_bits.shape[0], _p(out)))
    return out
