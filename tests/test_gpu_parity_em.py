"""GPU parity for the expert-major ("GEMM") receive layout: layout +
dispatch in one call, the cached-handle dispatch and the combine, through the
C ABI, against the oracle.

Bars: counts, group offsets, e4m3 bytes, bf16 rows, group-major scales,
source indices and weights (padding rows included) bit-exact; combine within
1 bf16 ulp and >= 99.9% bit-exact (100% expected: both sides add in
ascending expert id with RN fp32 adds).
"""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_get_03_gb300 import ep
from combine_ep_get_03_gb300 import workloads as wl
from harness import DEV, assert_bf16_close, dev, host_bits

pytestmark = pytest.mark.gpu


def _inputs(R, E, k, H, tpr, seed, mask=0.02, dup=0.0):
    g = wl.rng(seed)
    T = R * tpr
    idx, w = wl.route_uniform(g, T, E, k)
    idx = wl.mask_entries(g, idx, mask)
    if dup:
        sel = g.random(T) < dup
        idx[sel, k - 1] = idx[sel, 0]
    x = wl.normal_bf16(g, (T, H))
    return idx, w, x


def em_path(R, E, k, H, idx, w, x, fp8, align, y=None, num_sms=0, handle=None, cap=None, ids32=False):
    """Expert-major layout + dispatch (+ combine of y) through the ABI, each
    output against the oracle.  Returns (handle, oracle layout, dispatch ref)."""
    T = idx.shape[0]
    h = handle or ep.Handle(R, E, k, H, max(T // R, 1))
    if ids32:
        h.set_topk_idx_bits(32)
    L = oracle.em_layout(R, E, k, idx, align)
    rows = int(L["expert_offset"][-1])
    cap = rows if cap is None else cap
    ld = (max(cap, 1) + 3) // 4 * 4
    G = H // 128
    n = max(cap, 1)
    recv = torch.zeros((n, H), dtype=torch.uint8 if fp8 else torch.bfloat16, device=DEV)[:cap]
    scales = torch.full((G, ld), -7.0, dtype=torch.float32, device=DEV) if fp8 else None
    src = torch.full((n,), -7, dtype=torch.int32, device=DEV)[:cap]
    wts = torch.full((n,), -7.0, dtype=torch.float32, device=DEV)[:cap]
    h.em_layout_and_dispatch(dev(idx.astype(np.int32) if ids32 else idx), dev(x), dev(w),
                             ep.EP_FP8_E4M3 if fp8 else ep.EP_BF16, align, recv, scales, recv_src_idx=src,
                             recv_weights=wts, num_sms=num_sms)
    counts, offsets, st = h.em_get_layout(check=False)
    assert np.array_equal(counts, L["num_recv_per_expert"]), "num_recv_tokens_per_expert"
    assert np.array_equal(offsets, L["expert_offset"]), "expert_offset"
    ref, rst = oracle.em_dispatch(R, E, k, x, idx, w, fp8=fp8, align=align, capacity_rows=cap, scales_ld=ld)
    assert st == (ep.EP_OK if rst == oracle.OK else ep.EP_ERR_CAPACITY)
    used = min(rows, cap)
    real = ref["recv_src_idx"][:used] >= 0
    got_src = src.cpu().numpy()[:used]
    assert np.array_equal(got_src, ref["recv_src_idx"][:used]), "recv_src_idx (padding -1)"
    assert np.array_equal(wts.cpu().numpy()[:used].view(np.uint32), ref["recv_weights"][:used].view(np.uint32)), \
        "recv_weights (padding 0)"
    gx = recv.cpu().numpy() if fp8 else host_bits(recv)
    assert np.array_equal(gx[:used][real], ref["recv_x"][:used][real]), "recv_x rows"
    if fp8:
        gs = scales.cpu().numpy()
        assert np.array_equal(gs[:, :used][:, real].view(np.uint32), ref["recv_scales"][:, :used][:, real].view(np.uint32)), \
            "group-major scales"
    if y is not None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
        h.em_combine(dev(y), out, num_sms=num_sms)
        frac = assert_bf16_close(host_bits(out), oracle.em_combine(R, E, k, idx, align, y), "em combine")
        assert frac == 1.0
    status = h.get_device_status()
    assert status == (ep.EP_OK if rst == oracle.OK else ep.EP_ERR_CAPACITY)
    return h, L, ref


@pytest.mark.parametrize("name,align", [("tiny_bf16", 1), ("v3_ep8", 128), ("v3_ep8_group_limited", 64),
                                        ("ll_decode_ep8", 8), ("large_ep64_bwd", 32)])
def test_em_workloads(name, align):
    w_ = wl.WORKLOADS[name]
    x, idx, wts = wl.make_inputs(w_)
    rows = int(oracle.em_layout(w_.R, w_.E, w_.k, idx, align)["expert_offset"][-1])
    y = wl.normal_bf16(wl.rng(w_.seed + 300), (rows, w_.H))
    h, L, _ = em_path(w_.R, w_.E, w_.k, w_.H, idx, wts, x, fp8=w_.fp8, align=align, y=y)
    # the cached handle serves a BF16 dispatch of gradients afterwards
    g = wl.normal_bf16(wl.rng(w_.seed + 301), (w_.T, w_.H), 1e-2)
    recv = torch.empty((rows, w_.H), dtype=torch.bfloat16, device=DEV)
    src = torch.full((rows,), -7, dtype=torch.int32, device=DEV)
    h.em_dispatch(dev(g), dev(wts), ep.EP_BF16, recv, recv_src_idx=src)
    ref, _ = oracle.em_dispatch(w_.R, w_.E, w_.k, g, idx, wts, fp8=False, align=align)
    real = ref["recv_src_idx"] >= 0
    assert np.array_equal(src.cpu().numpy(), ref["recv_src_idx"])
    assert np.array_equal(host_bits(recv)[real], ref["recv_x"][real])
    assert h.get_device_status() == ep.EP_OK
    h.close()


EDGE = [(4, 16, 2, 256, 16, 0.0, 0.0, 1), (8, 64, 8, 1024, 64, 0.05, 0.2, 16), (3, 12, 4, 384, 33, 0.3, 0.3, 4),
        (64, 256, 8, 512, 8, 0.02, 0.0, 32), (8, 16, 8, 128, 5, 0.0, 0.5, 128), (2, 4096, 8, 128, 64, 0.0, 0.0, 2)]


@pytest.mark.parametrize("case", EDGE, ids=[f"R{c[0]}E{c[1]}k{c[2]}H{c[3]}t{c[4]}a{c[7]}" for c in EDGE])
def test_em_edge_shapes(case):
    R, E, k, H, tpr, mask, dup, align = case
    idx, w, x = _inputs(R, E, k, H, tpr, seed=sum(case[:5]), mask=mask, dup=dup)
    rows = int(oracle.em_layout(R, E, k, idx, align)["expert_offset"][-1])
    y = wl.normal_bf16(wl.rng(5), (rows, H))
    h = ep.Handle(R, E, k, H, tpr)
    for fp8 in (False, True):
        em_path(R, E, k, H, idx, w, x, fp8=fp8, align=align, y=y, handle=h)
    h.close()


@pytest.mark.parametrize("num_sms", [1, 7])
def test_em_few_sms_and_int32_ids(num_sms):
    R, E, k, H, tpr = 8, 64, 8, 1024, 48
    idx, w, x = _inputs(R, E, k, H, tpr, seed=80 + num_sms, dup=0.1)
    rows = int(oracle.em_layout(R, E, k, idx, 16)["expert_offset"][-1])
    y = wl.normal_bf16(wl.rng(81), (rows, H))
    h, _, _ = em_path(R, E, k, H, idx, w, x, fp8=True, align=16, y=y, num_sms=num_sms, ids32=True)
    h.close()


def test_em_falls_back_to_separate_kernels():
    """More than 4096 (token, k) entries per SM: routing kernel, offsets
    kernel and scatter give the same results."""
    R, E, k, H, tpr = 8, 64, 8, 128, 10240
    idx, w, x = _inputs(R, E, k, H, tpr, seed=71)
    rows = int(oracle.em_layout(R, E, k, idx, 32)["expert_offset"][-1])
    y = wl.normal_bf16(wl.rng(72), (rows, H))
    h, _, _ = em_path(R, E, k, H, idx, w, x, fp8=True, align=32, y=y)
    h.close()


def test_em_capacity_overflow_is_latched_and_in_bounds():
    R, E, k, H, tpr, align = 4, 16, 2, 256, 16, 4
    idx, w, x = _inputs(R, E, k, H, tpr, seed=73)
    rows = int(oracle.em_layout(R, E, k, idx, align)["expert_offset"][-1])
    for fp8 in (False, True):
        h, _, _ = em_path(R, E, k, H, idx, w, x, fp8=fp8, align=align, cap=rows - 11)
        h.close()


def test_em_zero_tokens_and_state_errors():
    R, E, k, H = 4, 16, 2, 256
    h = ep.Handle(R, E, k, H, 8)
    out = torch.empty((1, H), dtype=torch.bfloat16, device=DEV)
    L_ = ep.lib()
    assert L_.ep_em_combine(h.ptr, None, 0, out.data_ptr(), 0, None) == ep.EP_ERR_STATE
    assert L_.ep_em_get_layout(h.ptr, None, None, None) == ep.EP_ERR_STATE
    idx = torch.empty((0, k), dtype=torch.int64, device=DEV)
    x = torch.empty((0, H), dtype=torch.bfloat16, device=DEV)
    recv = torch.empty((0, H), dtype=torch.bfloat16, device=DEV)
    h.em_layout_and_dispatch(idx, x, None, ep.EP_BF16, 4, recv)
    counts, offsets, st = h.em_get_layout()
    assert not counts.any() and not offsets.any() and st == ep.EP_OK
    # bad alignment, scales_ld below capacity
    assert L_.ep_em_layout_and_dispatch(h.ptr, idx.data_ptr(), 0, x.data_ptr(), None, ep.EP_BF16, 0, None, None, 0,
                                        0, None, None, 0, None) == ep.EP_ERR_INVALID_ARG
    r8 = torch.empty((8, H), dtype=torch.uint8, device=DEV)
    sc = torch.empty((H // 128, 8), dtype=torch.float32, device=DEV)
    assert L_.ep_em_layout_and_dispatch(h.ptr, idx.data_ptr(), 0, x.data_ptr(), None, ep.EP_FP8_E4M3, 4,
                                        r8.data_ptr(), sc.data_ptr(), 6, 8, None, None, 0,
                                        None) == ep.EP_ERR_INVALID_ARG
    h.close()
