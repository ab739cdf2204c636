"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on
the five seeded workloads at full size, plus edge cases.

Bar: layout, counts, offsets, permutation, metadata, e4m3 bytes and fp32
scales bit-exact; combine within 1 bf16 ulp with >= 99.9% bit-exact.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_get_03_gb300 import ep
from combine_ep_get_03_gb300 import workloads as wl

from harness import (DEV, assert_bf16_close, check_layout, compare_dispatch, dev, fused_path, host_bits, ll_path,
                     normal_path, run_combine, run_dispatch)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    yield
    torch.cuda.synchronize()


# ------------------------------------------------------------ workloads

def test_tiny_bf16_workload():
    w_ = wl.WORKLOADS["tiny_bf16"]
    x, idx, wts = wl.make_inputs(w_)
    h, L, ref, _ = normal_path(w_.R, w_.E, w_.k, w_.H, idx, wts, x, fp8=False)
    # combine input: the dispatched rows scaled by 0.5 in bf16
    y = wl.f32_to_bf16_bits(wl.bf16_bits_to_f32(ref["recv_x"]) * np.float32(0.5))
    got = run_combine(h, y)
    assert np.array_equal(got, oracle.combine(w_.R, w_.E, w_.k, idx, y))
    h.close()


@pytest.mark.parametrize("name", ["v3_ep8", "v3_ep8_group_limited"])
def test_v3_shaped_workloads(name):
    w_ = wl.WORKLOADS[name]
    x, idx, wts = wl.make_inputs(w_)
    L = oracle.layout(w_.R, w_.E, w_.k, idx)
    P = int(L["rank_offset"][-1])
    y = wl.expert_outputs(w_, P)
    h, _, _, frac = normal_path(w_.R, w_.E, w_.k, w_.H, idx, wts, x, fp8=True, y=y)
    assert frac == 1.0
    h.close()


def test_ll_decode_workload():
    w_ = wl.WORKLOADS["ll_decode_ep8"]
    x, idx, wts = wl.make_inputs(w_)
    h, _, frac = ll_path(w_.R, w_.E, w_.k, w_.H, idx, wts, x, fp8=True, y_seed=w_.seed + 7)
    assert frac == 1.0
    h.close()


def test_large_ep_backward_workload():
    """Forward FP8 dispatch + combine, then the backward on the same handle:
    BF16 dispatch of grad_out (combine's adjoint) and a combine of the expert
    gradients (dispatch's adjoint) -- no new layout."""
    w_ = wl.WORKLOADS["large_ep64_bwd"]
    x, idx, wts = wl.make_inputs(w_)
    L = oracle.layout(w_.R, w_.E, w_.k, idx)
    P = int(L["rank_offset"][-1])
    y = wl.expert_outputs(w_, P)
    h, _, _, frac = normal_path(w_.R, w_.E, w_.k, w_.H, idx, wts, x, fp8=True, y=y)
    assert frac == 1.0
    g = wl.rng(w_.seed + 200)
    grad_out = wl.normal_bf16(g, (w_.T, w_.H), w_.grad_sigma)
    got = run_dispatch(h, dev(grad_out), dev(wts), False, P)
    ref, _ = oracle.dispatch(w_.R, w_.E, w_.k, grad_out, idx, wts, fp8=False)
    compare_dispatch(got, ref, False, P)
    grad_recv = wl.normal_bf16(g, (P, w_.H), w_.grad_sigma)
    gx = run_combine(h, grad_recv)
    assert assert_bf16_close(gx, oracle.combine(w_.R, w_.E, w_.k, idx, grad_recv), "grad combine") == 1.0
    assert h.get_device_status() == ep.EP_OK
    h.close()


# ------------------------------------------------------------ edge cases

EDGE = [
    # R, E, k, H, tokens_per_rank, mask, dup
    (3, 12, 6, 640, 100, 0.05, 0.2),   # k not a power of two, ragged H and chunks
    (1, 8, 1, 128, 1, 0.0, 0.0),       # one rank, one token, top-1
    (64, 64, 8, 256, 3, 0.02, 0.0),    # one expert per rank, 3 tokens per rank
    (2, 64, 32, 384, 40, 0.1, 0.0),    # top-32: a whole warp per token
    (8, 256, 8, 7168, 33, 0.01, 0.05), # V3 hidden, odd token count
    (5, 40, 4, 1024, 257, 0.3, 0.3),   # heavy masking and duplicates
    (2, 4, 2, 40960, 4, 0.0, 0.0),     # rows too long for the bulk-copy staging: register kernels
]


def _edge_inputs(R, E, k, H, tpr, mask, dup, seed):
    g = wl.rng(seed)
    T = R * tpr
    idx, w = wl.route_uniform(g, T, E, k)
    if mask:
        idx = wl.mask_entries(g, idx, mask)
    if dup:
        sel = g.random(T) < dup
        idx[sel, k - 1] = idx[sel, 0]
    x = wl.normal_bf16(g, (T, H))
    return idx, w, x


@pytest.mark.parametrize("case", EDGE, ids=[f"R{c[0]}E{c[1]}k{c[2]}H{c[3]}t{c[4]}" for c in EDGE])
def test_edge_shapes_all_steps(case):
    R, E, k, H, tpr, mask, dup = case
    idx, w, x = _edge_inputs(R, E, k, H, tpr, mask, dup, seed=sum(case[:5]))
    L = oracle.layout(R, E, k, idx)
    P = int(L["rank_offset"][-1])
    y = wl.normal_bf16(wl.rng(3), (P, H))
    h = ep.Handle(R, E, k, H, tpr)
    for fp8 in (False, True):
        normal_path(R, E, k, H, idx, w, x, fp8=fp8, y=y, handle=h)
    for fp8 in (False, True):
        ll_path(R, E, k, H, idx, w, x, fp8=fp8, y_seed=5, handle=h)
    h.close()


@pytest.mark.parametrize("H", [512, 1024])
def test_long_scatter_pipelines(H):
    """Many tokens per warp, so every row buffer and barrier of the bulk-copy
    scatter cycles several times (BF16 and FP8, normal and low latency)."""
    R, E, k, tpr = 8, 64, 4, 2048
    idx, w, x = _edge_inputs(R, E, k, H, tpr, 0.01, 0.05, seed=H)
    L = oracle.layout(R, E, k, idx)
    y = wl.normal_bf16(wl.rng(9), (int(L["rank_offset"][-1]), H))
    h = ep.Handle(R, E, k, H, tpr)
    for fp8 in (False, True):
        normal_path(R, E, k, H, idx, w, x, fp8=fp8, y=y, handle=h)
        normal_path(R, E, k, H, idx, w, x, fp8=fp8, handle=h, num_sms=7)
        ll_path(R, E, k, H, idx, w, x, fp8=fp8, y_seed=3, handle=h)
    h.close()


# ------------------------------------------------------------ fused layout + dispatch

@pytest.mark.parametrize("name", ["tiny_bf16", "v3_ep8", "v3_ep8_group_limited", "large_ep64_bwd"])
def test_fused_layout_dispatch_workloads(name):
    w_ = wl.WORKLOADS[name]
    x, idx, wts = wl.make_inputs(w_)
    P = int(oracle.layout(w_.R, w_.E, w_.k, idx)["rank_offset"][-1])
    y = wl.expert_outputs(w_, P)
    h, _, _, frac = fused_path(w_.R, w_.E, w_.k, w_.H, idx, wts, x, fp8=w_.fp8, y=y)
    assert frac == 1.0
    # the handle serves a cached-handle (backward) dispatch afterwards
    g = wl.normal_bf16(wl.rng(w_.seed + 200), (w_.T, w_.H), 1e-2)
    got = run_dispatch(h, dev(g), dev(wts), False, P)
    ref, _ = oracle.dispatch(w_.R, w_.E, w_.k, g, idx, wts, fp8=False)
    compare_dispatch(got, ref, False, P)
    h.close()


@pytest.mark.parametrize("case", EDGE, ids=[f"R{c[0]}E{c[1]}k{c[2]}H{c[3]}t{c[4]}" for c in EDGE])
def test_fused_layout_dispatch_edge_shapes(case):
    R, E, k, H, tpr, mask, dup = case
    idx, w, x = _edge_inputs(R, E, k, H, tpr, mask, dup, seed=sum(case[:5]) + 1)
    y = wl.normal_bf16(wl.rng(3), (int(oracle.layout(R, E, k, idx)["rank_offset"][-1]), H))
    h = ep.Handle(R, E, k, H, tpr)
    for fp8 in (False, True):
        fused_path(R, E, k, H, idx, w, x, fp8=fp8, y=y, handle=h)
    h.close()


@pytest.mark.parametrize("num_sms", [1, 7])
def test_fused_on_few_sms(num_sms):
    """One block (the grid barrier degenerates) and a handful of blocks."""
    R, E, k, H, tpr = 8, 64, 8, 1024, 48
    idx, w, x = _edge_inputs(R, E, k, H, tpr, 0.02, 0.1, seed=60 + num_sms)
    y = wl.normal_bf16(wl.rng(61), (int(oracle.layout(R, E, k, idx)["rank_offset"][-1]), H))
    h = ep.Handle(R, E, k, H, tpr)
    fused_path(R, E, k, H, idx, w, x, fp8=True, y=y, handle=h, num_sms=num_sms)
    ll_path(R, E, k, H, idx, w, x, fp8=True, y_seed=62, handle=h, num_sms=num_sms)
    h.close()


@pytest.mark.parametrize("num_sms", [152, 64, 24])
def test_fused_own_tokens_first_with_claims(num_sms):
    """Rank-major batches past the small-batch limit (the grid barrier):
    every block moves a ring of its own tokens first (destinations from its
    shared memory), then claims the rest -- none left at 7 tokens per block
    (152 SMs), 8 of 16 (64 SMs), 35 of 43 (24 SMs). Rows, metadata and the
    combine of them against the oracle; then the low-latency dispatch on the
    same handle (the per-entry routing with the same rows order)."""
    R, E, k, H, tpr = 8, 256, 8, 1024, 128
    idx, w, x = _edge_inputs(R, E, k, H, tpr, 0.02, 0.05, seed=90 + num_sms)
    y = wl.normal_bf16(wl.rng(91), (int(oracle.layout(R, E, k, idx)["rank_offset"][-1]), H))
    h = ep.Handle(R, E, k, H, tpr)
    for fp8 in (True, False):
        fused_path(R, E, k, H, idx, w, x, fp8=fp8, y=y, handle=h, num_sms=num_sms)
    ll_path(R, E, k, H, idx, w, x, fp8=True, y_seed=92, handle=h, num_sms=num_sms)
    h.close()


@pytest.mark.parametrize("num_sms", [16, 15, 152])
def test_ll_own_rows_boundary(num_sms):
    """Small low-latency batches move each block's own tokens when they fit
    its ring (16 SMs: exactly 8 tokens per block, one per consumer warp) and
    claim tokens otherwise (15 SMs: 9 per block); every block counts the ids
    of the tokens before its own. The same results either way."""
    R, E, k, H, tpr = 8, 64, 8, 1024, 16
    idx, w, x = _edge_inputs(R, E, k, H, tpr, 0.03, 0.1, seed=80 + num_sms)
    h = ep.Handle(R, E, k, H, tpr)
    for fp8 in (True, False):
        ll_path(R, E, k, H, idx, w, x, fp8=fp8, y_seed=81, handle=h, num_sms=num_sms)
    h.close()


@pytest.mark.parametrize("case", [(128, 128, 4, 128, 2), (8, 64, 8, 128, 10240)],
                         ids=["R128_layout_kernel", "T81920_routing_kernels"])
def test_fused_falls_back_to_separate_kernels(case):
    """More ranks than a 64-bit mask holds, or more than 4096 (token, k)
    entries per SM: the same results through the separate kernels."""
    R, E, k, H, tpr = case
    idx, w, x = _edge_inputs(R, E, k, H, tpr, 0.02, 0.0, seed=sum(case))
    y = wl.normal_bf16(wl.rng(70), (int(oracle.layout(R, E, k, idx)["rank_offset"][-1]), H))
    h = ep.Handle(R, E, k, H, tpr)
    fused_path(R, E, k, H, idx, w, x, fp8=True, y=y, handle=h)
    ll_path(R, E, k, H, idx, w, x, fp8=True, y_seed=71, handle=h)
    h.close()


def test_zero_tokens():
    R, E, k, H = 4, 16, 2, 256
    h = ep.Handle(R, E, k, H, 8)
    idx = np.zeros((0, k), np.int64)
    ntpr = torch.full((R, R), 5, dtype=torch.int32, device=DEV)
    h.get_dispatch_layout(dev(idx), num_tokens_per_rank=ntpr)
    a, b, off, st = h.get_num_recv()
    assert st == ep.EP_OK and not a.any() and not b.any() and not off.any()
    assert not ntpr.any()
    x = torch.empty((0, H), dtype=torch.bfloat16, device=DEV)
    recv = torch.empty((0, H), dtype=torch.bfloat16, device=DEV)
    h.dispatch(x, None, ep.EP_BF16, recv)
    h.combine(recv, torch.empty((0, H), dtype=torch.bfloat16, device=DEV))
    assert h.get_device_status() == ep.EP_OK
    h.close()


def test_tokens_with_no_destination_combine_to_zero():
    R, E, k, H, tpr = 4, 16, 2, 256, 16
    idx, w, x = _edge_inputs(R, E, k, H, tpr, 0.0, 0.0, seed=12)
    idx[::3] = -1  # every third token fully masked
    L = oracle.layout(R, E, k, idx)
    y = wl.normal_bf16(wl.rng(4), (int(L["rank_offset"][-1]), H))
    h, _, _, _ = normal_path(R, E, k, H, idx, w, x, fp8=True, y=y)
    out = run_combine(h, y)
    assert not out[::3].any()
    h.close()


def test_repeated_layouts_on_one_handle():
    """The scan state is reused across calls (epoch-tagged, never cleared)."""
    R, E, k, H, tpr = 8, 64, 4, 512, 200
    h = ep.Handle(R, E, k, H, tpr)
    for rep in range(4):
        idx, w, x = _edge_inputs(R, E, k, H, tpr - rep * 37, 0.02, 0.0, seed=40 + rep)
        y = wl.normal_bf16(wl.rng(rep), (int(oracle.layout(R, E, k, idx)["rank_offset"][-1]), H))
        normal_path(R, E, k, H, idx, w, x, fp8=bool(rep % 2), y=y, handle=h)
        ll_path(R, E, k, H, idx, w, x, fp8=not rep % 2, y_seed=rep, handle=h)
    h.close()


@pytest.mark.parametrize("num_sms", [1, 24, 64])
def test_num_sms_does_not_change_results(num_sms):
    R, E, k, H, tpr = 8, 256, 8, 2048, 256
    idx, w, x = _edge_inputs(R, E, k, H, tpr, 0.01, 0.0, seed=77)
    y = wl.normal_bf16(wl.rng(78), (int(oracle.layout(R, E, k, idx)["rank_offset"][-1]), H))
    h, _, _, _ = normal_path(R, E, k, H, idx, w, x, fp8=True, y=y, num_sms=num_sms)
    h.close()


# ------------------------------------------------------------ errors

def test_bad_expert_id_is_latched():
    R, E, k, H, tpr = 4, 16, 2, 256, 32
    idx, w, x = _edge_inputs(R, E, k, H, tpr, 0.0, 0.0, seed=5)
    idx[7, 1] = E + 3
    idx[9, 0] = -5
    h = ep.Handle(R, E, k, H, tpr)
    h.get_dispatch_layout(dev(idx))
    _, _, off, st = h.get_num_recv(check=False)
    assert st == ep.EP_ERR_BAD_EXPERT
    assert h.get_device_status() == ep.EP_ERR_BAD_EXPERT
    assert h.get_device_status() == ep.EP_OK  # cleared
    # the bad entries were treated as masked
    fixed = idx.copy()
    fixed[7, 1] = -1
    fixed[9, 0] = -1
    assert np.array_equal(off, oracle.layout(R, E, k, fixed)["rank_offset"])
    h.close()


def test_capacity_overflow_is_latched_and_in_bounds():
    R, E, k, H, tpr = 4, 16, 4, 256, 32
    idx, w, x = _edge_inputs(R, E, k, H, tpr, 0.0, 0.0, seed=6)
    L = oracle.layout(R, E, k, idx)
    P = int(L["rank_offset"][-1])
    h = ep.Handle(R, E, k, H, tpr)
    check_layout(h, idx, L)
    cap = P - 11
    guard = torch.full((P, H), 0x5A, dtype=torch.uint8, device=DEV)
    scales = torch.full((P, H // 128), 7.0, dtype=torch.float32, device=DEV)
    h.dispatch(dev(x), dev(w), ep.EP_FP8_E4M3, guard[:cap], scales[:cap])
    assert h.get_device_status() == ep.EP_ERR_CAPACITY
    ref, st = oracle.dispatch(R, E, k, x, idx, w, fp8=True, capacity_rows=cap)
    assert st == oracle.CAPACITY
    got = guard.cpu().numpy()
    assert np.array_equal(got[:cap], ref["recv_x"][:cap])
    assert (got[cap:] == 0x5A).all(), "rows past the capacity were written"
    assert (scales[cap:].cpu().numpy() == 7.0).all()
    # combine with too few rows: latched, in bounds
    y = wl.normal_bf16(wl.rng(1), (cap, H))
    out = torch.empty((R * tpr, H), dtype=torch.bfloat16, device=DEV)
    h.combine(dev(y), out)
    assert h.get_device_status() == ep.EP_ERR_CAPACITY
    h.close()


def test_a_wait_that_cannot_complete_ends_with_a_timeout_status():
    """Failure detection without a fault: waits on a word that nothing sets
    and on an mbarrier with no arrivals give up after their poll limit, the
    kernel returns, the handle reports EP_ERR_TIMEOUT once, and the handle
    and context still compute correct results afterwards."""
    import time

    R, E, k, H, tpr = 4, 16, 2, 256, 32
    idx, w, x = _edge_inputs(R, E, k, H, tpr, 0.0, 0.0, seed=8)
    h = ep.Handle(R, E, k, H, tpr)
    t0 = time.perf_counter()
    h.check_wait_timeout()
    st = h.get_device_status()
    dt = time.perf_counter() - t0
    assert st == ep.EP_ERR_TIMEOUT
    assert dt < 30.0, f"the bounded waits took {dt:.1f} s"
    assert h.get_device_status() == ep.EP_OK  # cleared
    # the fused kernel's control words were reset and everything still works
    y = wl.normal_bf16(wl.rng(9), (int(oracle.layout(R, E, k, idx)["rank_offset"][-1]), H))
    fused_path(R, E, k, H, idx, w, x, fp8=True, y=y, handle=h)
    ll_path(R, E, k, H, idx, w, x, fp8=True, y_seed=9, handle=h)
    assert h.get_device_status() == ep.EP_OK
    h.close()


def test_argument_errors_are_synchronous():
    h = ep.Handle(4, 16, 2, 256, 8)
    with pytest.raises(ep.EPError) as e:
        ep.ep_dispatch(h.ptr, None, None, ep.EP_BF16, torch.empty((4, 256), dtype=torch.bfloat16, device=DEV))
    assert e.value.status == ep.EP_ERR_STATE
    with pytest.raises(ep.EPError) as e:
        h.get_dispatch_layout(dev(np.zeros((6, 2), np.int64)))  # 6 tokens over 4 ranks
    assert e.value.status == ep.EP_ERR_INVALID_ARG
    with pytest.raises(ep.EPError) as e:
        ep.ep_handle_create(4, 18, 2, 256, 8)  # experts not divisible by ranks
    assert e.value.status == ep.EP_ERR_INVALID_ARG
    h.close()


# ------------------------------------------------------------ formats

def test_e4m3_conversion_all_bf16_values():
    """Groups whose largest magnitude is 448 have 448/amax = 1 exactly, so
    the kernel's e4m3 conversion sees every finite bf16 value |v| <= 448
    unscaled; bytes must equal the oracle's encoder."""
    bits = np.arange(65536, dtype=np.uint32) << 16
    v = bits.view(np.float32)
    v = v[np.isfinite(v) & (np.abs(v) <= 448.0)]
    n_groups = -(-v.size // 127)
    pad = np.zeros(n_groups * 127, np.float32)
    pad[: v.size] = v
    groups = np.concatenate([np.full((n_groups, 1), 448.0, np.float32), pad.reshape(n_groups, 127)], axis=1)
    H = 128 * 16
    rows = -(-n_groups // 16)
    allg = np.zeros((rows * 16, 128), np.float32)
    allg[:n_groups] = groups
    allg[n_groups:, 0] = 448.0
    x = wl.f32_to_bf16_bits(allg.reshape(rows, H))
    R, E, k = 1, 1, 1
    idx = np.zeros((rows, 1), np.int64)
    w = np.ones((rows, 1), np.float32)
    h, _, ref, _ = normal_path(R, E, k, H, idx, w, x, fp8=True)
    # every scale is exactly 1
    assert np.all(ref["recv_scales"] == np.float32(1.0))
    h.close()


def test_ll_path_captures_in_a_cuda_graph():
    """Low-latency dispatch + combine have no host synchronisation and no
    allocation: capture once, replay, same bytes as an eager call."""
    R, E, k, H, tpr = 8, 64, 8, 1024, 16
    idx, w, x = _edge_inputs(R, E, k, H, tpr, 0.0, 0.0, seed=88)
    h = ep.Handle(R, E, k, H, tpr)
    M = h.M
    x_d, idx_d, w_d = dev(x), dev(idx), dev(w)
    recv = torch.zeros((E, M, H), dtype=torch.uint8, device=DEV)
    scales = torch.zeros((E, M, H // 128), dtype=torch.float32, device=DEV)
    y = torch.randn((E, M, H), device=DEV).to(torch.bfloat16)
    out_eager = torch.empty((R * tpr, H), dtype=torch.bfloat16, device=DEV)
    out_graph = torch.empty_like(out_eager)
    h.low_latency_dispatch(x_d, idx_d, ep.EP_FP8_E4M3, recv, scales)
    h.low_latency_combine(y, w_d, out_eager)
    recv_eager = recv.clone()
    scales_eager = scales.clone()
    recv.zero_()
    scales.zero_()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            h.low_latency_dispatch(x_d, idx_d, ep.EP_FP8_E4M3, recv, scales)
            h.low_latency_combine(y, w_d, out_graph)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(recv, recv_eager)
    assert torch.equal(scales, scales_eager)
    assert torch.equal(out_graph.view(torch.int16), out_eager.view(torch.int16))
    assert h.get_device_status() == ep.EP_OK
    h.close()


@pytest.mark.parametrize("num_sms", [0, 3])
def test_ll_capacity_overflow_and_bad_id_latched(num_sms):
    """Low-latency dispatch on a small batch (own rows on every SM, claims on
    3 SMs): one expert receives more entries than its M rows (duplicated
    ids), and one id is out of range. Both conditions are latched; the first
    M entries of the full expert land where the oracle puts them, the bad id
    counts as masked, and the combine of the dispatched rows matches the
    oracle's, which skips the entries that got no row."""
    R, E, k, H, tpr = 4, 16, 4, 256, 16
    T = R * tpr
    g = wl.rng(97 + num_sms)
    idx, w = wl.route_uniform(g, T, E, k)
    idx[:, :] = np.where(np.arange(T)[:, None] % 2 == 0, 5, idx)  # even tokens: all four entries on expert 5
    idx[3, 2] = E + 3
    x = wl.normal_bf16(g, (T, H))
    h = ep.Handle(R, E, k, H, tpr)
    M = h.M
    recv = torch.zeros((E, M, H), dtype=torch.uint8, device=DEV)
    scales = torch.zeros((E, M, H // 128), dtype=torch.float32, device=DEV)
    src = torch.full((E, M), -7, dtype=torch.int32, device=DEV)
    cnt = torch.full((E,), -7, dtype=torch.int32, device=DEV)
    h.low_latency_dispatch(dev(x), dev(idx), ep.EP_FP8_E4M3, recv, scales, recv_src_info=src, recv_count=cnt,
                           num_sms=num_sms)
    st = h.get_device_status()
    assert st in (ep.EP_ERR_BAD_EXPERT, ep.EP_ERR_CAPACITY)  # the first condition wins the latch
    fixed = idx.copy()
    fixed[3, 2] = -1
    ref, rst = oracle.ll_dispatch(R, E, k, M, x, fixed, fp8=True)
    assert rst == oracle.CAPACITY
    count = cnt.cpu().numpy()
    assert np.array_equal(count, ref["recv_count"])
    assert count[5] == M
    flat = np.concatenate([e * M + np.arange(c) for e, c in enumerate(count)]).astype(np.int64)
    fl = torch.from_numpy(flat).to(DEV)
    assert np.array_equal(recv.view(E * M, H)[fl].cpu().numpy(), ref["recv_x"].reshape(E * M, H)[flat])
    assert np.array_equal(src.view(-1)[fl].cpu().numpy(), ref["recv_src_info"].reshape(-1)[flat])
    y_host = np.zeros((E, M, H), np.uint16)
    y_host.reshape(E * M, H)[flat] = wl.normal_bf16(wl.rng(98), (flat.size, H))
    out = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    h.low_latency_combine(dev(y_host), dev(w), out, num_sms=num_sms)
    assert np.array_equal(host_bits(out), oracle.ll_combine(R, E, k, M, fixed, w, y_host))
    assert h.get_device_status() == ep.EP_OK
    h.close()
