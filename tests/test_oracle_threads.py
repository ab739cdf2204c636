"""The oracle's multi-threaded copy (used only to time the CPU baseline on all
host cores) gives byte-identical results to the single-threaded definitions:
the same per-token arithmetic, the token loop split into ranges."""
import numpy as np
import pytest

import oracle
from combine_ep_get_03_gb300 import workloads as wl

# (R, E, k, tokens per rank, H, mask fraction): masking, duplicates via a
# small E, a token count no thread count divides evenly
SHAPES = [(8, 64, 8, 37, 256, 0.05), (4, 16, 6, 25, 384, 0.2)]


def _inputs(R, E, k, tpr, H, mask, seed):
    T = R * tpr
    g = wl.rng(seed)
    idx, w = wl.route_uniform(g, T, E, k)
    idx = wl.mask_entries(g, idx, mask)
    if E <= 16:
        idx[::7, 1] = idx[::7, 0]  # duplicated expert ids inside a token
    return idx, w, wl.normal_bf16(g, (T, H))


@pytest.mark.parametrize("shape", SHAPES)
def test_threaded_oracle_is_byte_identical(shape):
    R, E, k, tpr, H, mask = shape
    idx, w, x = _inputs(R, E, k, tpr, H, mask, 77)
    T = idx.shape[0]
    n_cores = oracle.threads_available()
    assert n_cores >= 1
    for threads in sorted({1, 3, n_cores, T + 5}):
        for fp8 in (False, True):
            a, sa = oracle.dispatch(R, E, k, x, idx, w, fp8=fp8)
            b, sb = oracle.dispatch(R, E, k, x, idx, w, fp8=fp8, threads=threads)
            assert sa == sb
            for key in a:
                if a[key] is not None:
                    assert a[key].tobytes() == b[key].tobytes(), (threads, fp8, key)
        P = int(oracle.layout(R, E, k, idx)["rank_offset"][-1])
        y = wl.normal_bf16(wl.rng(78), (P, H))
        assert oracle.combine(R, E, k, idx, y).tobytes() == oracle.combine(R, E, k, idx, y, threads=threads).tobytes()
        d, _ = oracle.dispatch(R, E, k, x, idx, w, fp8=True)
        rw = d["recv_topk_weights"]
        o1, c1 = oracle.combine_ex(R, E, k, idx, d["recv_x"], y_scales=d["recv_scales"], recv_topk_weights=rw)
        o2, c2 = oracle.combine_ex(R, E, k, idx, d["recv_x"], y_scales=d["recv_scales"], recv_topk_weights=rw,
                                   threads=threads)
        assert o1.tobytes() == o2.tobytes() and c1.tobytes() == c2.tobytes()
        M = T
        for fp8 in (False, True):
            a, sa = oracle.ll_dispatch(R, E, k, M, x, idx, fp8=fp8)
            b, sb = oracle.ll_dispatch(R, E, k, M, x, idx, fp8=fp8, threads=threads)
            assert sa == sb
            for key in a:
                if a[key] is not None:
                    assert a[key].tobytes() == b[key].tobytes(), (threads, fp8, key)
        y_ll = wl.normal_bf16(wl.rng(79), (E, M, H))
        assert oracle.ll_combine(R, E, k, M, idx, w, y_ll).tobytes() == \
            oracle.ll_combine(R, E, k, M, idx, w, y_ll, threads=threads).tobytes()


def test_threaded_oracle_reports_capacity_like_the_plain_one():
    R, E, k, tpr, H = 4, 16, 4, 16, 128
    idx, w, x = _inputs(R, E, k, tpr, H, 0.0, 80)
    a, sa = oracle.dispatch(R, E, k, x, idx, w, fp8=True, capacity_rows=10)
    b, sb = oracle.dispatch(R, E, k, x, idx, w, fp8=True, capacity_rows=10, threads=4)
    assert sa == sb == oracle.CAPACITY
    assert a["recv_x"].tobytes() == b["recv_x"].tobytes()
    a, sa = oracle.ll_dispatch(R, E, k, 3, x, idx, fp8=False)
    b, sb = oracle.ll_dispatch(R, E, k, 3, x, idx, fp8=False, threads=4)
    assert sa == sb == oracle.CAPACITY
    assert a["recv_x"].tobytes() == b["recv_x"].tobytes() and a["slot"].tobytes() == b["slot"].tobytes()
