"""Helpers for the GPU parity tests: run each hot-path step through the
C-ABI library (via the ctypes binding) and compare with the CPU oracle on
the same seeded inputs.

Tolerances: layout, slots, permutation, metadata, e4m3 bytes and fp32
scales are compared bit for bit; combine outputs must be within 1 bf16 ulp
with at least 99.9% of elements bit-identical (both sides sum in the same
order with the same IEEE operations, so 100% is expected and reported).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from combine_ep_get_03_gb300 import ep
from combine_ep_get_03_gb300 import workloads as wl

DEV = "cuda:0"


def dev(a: np.ndarray, dtype=None) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16)).to(DEV)
        return t.view(torch.bfloat16) if dtype is None else t.view(dtype)
    t = torch.from_numpy(a).to(DEV)
    return t if dtype is None else t.view(dtype)


def host_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 numpy bits."""
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def assert_bf16_close(got: np.ndarray, ref: np.ndarray, what: str, min_exact: float = 0.999) -> float:
    """Within 1 bf16 ulp everywhere and >= min_exact bit-identical."""
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if got.size == 0:
        return 1.0
    exact = got == ref
    frac = float(exact.mean())
    g = wl.bf16_bits_to_f32(got).astype(np.float64)
    r = wl.bf16_bits_to_f32(ref).astype(np.float64)
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(r), 2.0 ** -126))) - 7)
    bad = ~exact & (np.abs(g - r) > ulp)
    assert not bad.any(), f"{what}: {int(bad.sum())} elements beyond 1 bf16 ulp"
    assert frac >= min_exact, f"{what}: only {frac:.6f} bit-exact"
    return frac


def check_layout(h: ep.Handle, idx: np.ndarray, ref_layout=None):
    """Run ep_get_dispatch_layout; compare every output bit for bit."""
    R, E = h.R, h.E
    T = idx.shape[0]
    ntpr = torch.full((R, R), -9, dtype=torch.int32, device=DEV)
    ntpe = torch.full((R, E), -9, dtype=torch.int32, device=DEV)
    itr = torch.zeros((T, R), dtype=torch.bool, device=DEV)
    h.get_dispatch_layout(dev(idx), num_tokens_per_rank=ntpr, num_tokens_per_expert=ntpe, is_token_in_rank=itr)
    per_rank, per_expert, offset, st = h.get_num_recv()
    L = ref_layout if ref_layout is not None else oracle.layout(R, E, h.k, idx)
    assert np.array_equal(ntpr.cpu().numpy(), L["num_tokens_per_rank"]), "num_tokens_per_rank"
    assert np.array_equal(ntpe.cpu().numpy(), L["num_tokens_per_expert"]), "num_tokens_per_expert"
    assert np.array_equal(itr.cpu().numpy(), L["is_token_in_rank"]), "is_token_in_rank"
    assert np.array_equal(per_rank, L["num_recv_per_rank"]), "num_recv_tokens_per_rank"
    assert np.array_equal(per_expert, L["num_recv_per_expert"]), "num_recv_tokens_per_expert"
    assert np.array_equal(offset, L["rank_offset"]), "rank_offset"
    return L


def run_dispatch(h: ep.Handle, x_d, w_d, fp8: bool, P: int, cap: int | None = None, num_sms: int = 0):
    cap = P if cap is None else cap
    H, k = h.H, h.k
    rows = max(cap, 1)
    out = dict(
        recv_x=torch.empty((rows, H), dtype=torch.uint8 if fp8 else torch.bfloat16, device=DEV)[:cap],
        recv_scales=torch.empty((rows, H // 128), dtype=torch.float32, device=DEV)[:cap] if fp8 else None,
        recv_src_idx=torch.full((rows,), -7, dtype=torch.int32, device=DEV)[:cap],
        recv_topk_idx=torch.full((rows, k), -7, dtype=torch.int32, device=DEV)[:cap],
        recv_topk_weights=torch.full((rows, k), -7.0, dtype=torch.float32, device=DEV)[:cap],
    )
    h.dispatch(x_d, w_d, ep.EP_FP8_E4M3 if fp8 else ep.EP_BF16, out["recv_x"], out["recv_scales"],
               recv_src_idx=out["recv_src_idx"], recv_topk_idx=out["recv_topk_idx"],
               recv_topk_weights=out["recv_topk_weights"], num_sms=num_sms)
    return out


def compare_dispatch(got: dict, ref: dict, fp8: bool, rows: int):
    rx = got["recv_x"].cpu().numpy() if fp8 else host_bits(got["recv_x"])
    assert np.array_equal(rx[:rows], ref["recv_x"][:rows]), "recv_x bytes"
    if fp8:
        assert np.array_equal(got["recv_scales"].cpu().numpy()[:rows].view(np.uint32),
                              ref["recv_scales"][:rows].view(np.uint32)), "recv_scales bits"
    assert np.array_equal(got["recv_src_idx"].cpu().numpy()[:rows], ref["recv_src_idx"][:rows]), "recv_src_idx"
    assert np.array_equal(got["recv_topk_idx"].cpu().numpy()[:rows], ref["recv_topk_idx"][:rows]), "recv_topk_idx"
    assert np.array_equal(got["recv_topk_weights"].cpu().numpy()[:rows].view(np.uint32),
                          ref["recv_topk_weights"][:rows].view(np.uint32)), "recv_topk_weights"


def run_combine(h: ep.Handle, y_bits: np.ndarray, num_sms: int = 0) -> np.ndarray:
    T = h.T
    out = torch.empty((T, h.H), dtype=torch.bfloat16, device=DEV)
    h.combine(dev(y_bits), out, num_sms=num_sms)
    return host_bits(out)


def normal_path(R, E, k, H, idx, w, x, fp8, y=None, num_sms=0, handle=None):
    """Layout + dispatch (+ combine of y) through the ABI, each step checked
    against the oracle.  Returns (handle, layout, dispatch result, exact fraction)."""
    T = idx.shape[0]
    h = handle or ep.Handle(R, E, k, H, max(T // R, 1))
    L = check_layout(h, idx)
    P = int(L["rank_offset"][-1])
    got = run_dispatch(h, dev(x), dev(w), fp8, P, num_sms=num_sms)
    ref, st = oracle.dispatch(R, E, k, x, idx, w, fp8=fp8)
    assert st == oracle.OK
    compare_dispatch(got, ref, fp8, P)
    frac = None
    if y is not None:
        comb = run_combine(h, y, num_sms=num_sms)
        frac = assert_bf16_close(comb, oracle.combine(R, E, k, idx, y), "combine")
    assert h.get_device_status() == ep.EP_OK
    return h, L, ref, frac


def ll_path(R, E, k, H, idx, w, x, fp8, y_seed=None, num_sms=0, handle=None):
    """Low-latency dispatch (+ weighted combine of synthetic expert outputs)
    through the ABI, checked against the oracle on the filled rows."""
    T = idx.shape[0]
    h = handle or ep.Handle(R, E, k, H, max(T // R, 1))
    M = h.M
    G = H // 128
    recv = torch.empty((E, M, H), dtype=torch.uint8 if fp8 else torch.bfloat16, device=DEV)
    scales = torch.empty((E, M, G), dtype=torch.float32, device=DEV) if fp8 else None
    src = torch.full((E, M), -7, dtype=torch.int32, device=DEV)
    cnt = torch.full((E,), -7, dtype=torch.int32, device=DEV)
    h.low_latency_dispatch(dev(x), dev(idx), ep.EP_FP8_E4M3 if fp8 else ep.EP_BF16, recv, scales,
                           recv_src_info=src, recv_count=cnt, num_sms=num_sms)
    ref, st = oracle.ll_dispatch(R, E, k, M, x, idx, fp8=fp8)
    assert st == oracle.OK
    count = cnt.cpu().numpy()
    assert np.array_equal(count, ref["recv_count"]), "recv_count"
    flat = np.concatenate([e * M + np.arange(c) for e, c in enumerate(count)]).astype(np.int64)
    fl = torch.from_numpy(flat).to(DEV)
    got_x = recv.view(E * M, H)[fl]
    ref_x = ref["recv_x"].reshape(E * M, H)[flat]
    assert np.array_equal(got_x.cpu().numpy() if fp8 else host_bits(got_x), ref_x), "ll recv_x"
    if fp8:
        assert np.array_equal(scales.view(E * M, G)[fl].cpu().numpy().view(np.uint32),
                              ref["recv_scales"].reshape(E * M, G)[flat].view(np.uint32)), "ll recv_scales"
    assert np.array_equal(src.view(-1)[fl].cpu().numpy(), ref["recv_src_info"].reshape(-1)[flat]), "ll src_info"
    frac = None
    if y_seed is not None:
        # synthetic expert outputs on the filled rows only (the rest is never read)
        y_host = np.zeros((E, M, H), np.uint16)
        y_host.reshape(E * M, H)[flat] = wl.normal_bf16(wl.rng(y_seed), (flat.size, H))
        y_dev = torch.empty((E, M, H), dtype=torch.bfloat16, device=DEV)
        y_dev.view(E * M, H)[fl] = dev(y_host.reshape(E * M, H)[flat])
        out = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
        h.low_latency_combine(y_dev, dev(w), out, num_sms=num_sms)
        frac = assert_bf16_close(host_bits(out), oracle.ll_combine(R, E, k, M, idx, w, y_host), "ll combine")
    assert h.get_device_status() == ep.EP_OK
    return h, ref, frac


def fused_path(R, E, k, H, idx, w, x, fp8, y=None, num_sms=0, handle=None, cap=None):
    """ep_layout_and_dispatch through the ABI: the handle's layout state
    (counts, offsets, and -- through combine -- the destination rows) and the
    dispatch outputs, each against the oracle."""
    T = idx.shape[0]
    h = handle or ep.Handle(R, E, k, H, max(T // R, 1))
    L = oracle.layout(R, E, k, idx)
    P = int(L["rank_offset"][-1])
    cap = P if cap is None else cap
    rows = max(cap, 1)
    got = dict(
        recv_x=torch.empty((rows, H), dtype=torch.uint8 if fp8 else torch.bfloat16, device=DEV)[:cap],
        recv_scales=torch.empty((rows, H // 128), dtype=torch.float32, device=DEV)[:cap] if fp8 else None,
        recv_src_idx=torch.full((rows,), -7, dtype=torch.int32, device=DEV)[:cap],
        recv_topk_idx=torch.full((rows, k), -7, dtype=torch.int32, device=DEV)[:cap],
        recv_topk_weights=torch.full((rows, k), -7.0, dtype=torch.float32, device=DEV)[:cap],
    )
    h.layout_and_dispatch(dev(idx), dev(x), dev(w), ep.EP_FP8_E4M3 if fp8 else ep.EP_BF16, got["recv_x"],
                          got["recv_scales"], recv_src_idx=got["recv_src_idx"], recv_topk_idx=got["recv_topk_idx"],
                          recv_topk_weights=got["recv_topk_weights"], num_sms=num_sms)
    per_rank, per_expert, offset, st = h.get_num_recv()
    assert np.array_equal(per_rank, L["num_recv_per_rank"]), "num_recv_tokens_per_rank"
    assert np.array_equal(per_expert, L["num_recv_per_expert"]), "num_recv_tokens_per_expert"
    assert np.array_equal(offset, L["rank_offset"]), "rank_offset"
    ref, st = oracle.dispatch(R, E, k, x, idx, w, fp8=fp8)
    compare_dispatch(got, ref, fp8, P)
    frac = None
    if y is not None:
        comb = run_combine(h, y, num_sms=num_sms)
        frac = assert_bf16_close(comb, oracle.combine(R, E, k, idx, y), "combine after fused dispatch")
    assert h.get_device_status() == ep.EP_OK
    return h, L, ref, frac
