"""GPU parity for the general combine (e4m3 input, the top-k weights'
reduction) and for int32 top-k ids, through the C ABI, against the oracle.

Bars: e4m3 combine output within 1 bf16 ulp and >= 99.9% bit-exact (both
sides take decode * scale as one fp32 multiply and add in ascending rank
order, so 100% is expected); combined top-k weights bit-exact; everything
routed from int32 ids bit-identical to the int64 run's oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_get_03_gb300 import ep
from combine_ep_get_03_gb300 import workloads as wl
from harness import DEV, assert_bf16_close, dev, fused_path, host_bits, ll_path, normal_path, run_dispatch

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


CASES = [(4, 16, 2, 256, 16), (8, 64, 8, 1024, 64), (8, 256, 8, 7168, 96), (64, 256, 8, 512, 8), (3, 12, 4, 384, 33),
         (16, 64, 16, 1536, 12)]


@pytest.mark.parametrize("case", CASES, ids=[f"R{c[0]}E{c[1]}k{c[2]}H{c[3]}t{c[4]}" for c in CASES])
def test_combine_fp8_input_and_weights(case):
    R, E, k, H, tpr = case
    idx, w, x = _inputs(R, E, k, H, tpr, seed=sum(case))
    h, L, ref, _ = normal_path(R, E, k, H, idx, w, x, fp8=True)
    P = int(L["rank_offset"][-1])
    T = idx.shape[0]
    # e4m3 expert outputs: the dispatched rows themselves, then random codes
    # and scales (NaN codes excluded)
    g = wl.rng(7 + R)
    q_rand = g.integers(0, 256, (P, H), dtype=np.uint8)
    q_rand[(q_rand & 0x7F) == 0x7F] = 0
    s_rand = (g.random((P, H // 128)) * 3 + 1e-3).astype(np.float32)
    rw = (g.random((P, k)) - 0.5).astype(np.float32)
    for q, s in ((ref["recv_x"][:P], ref["recv_scales"][:P]), (q_rand, s_rand)):
        out = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
        cw = torch.full((T, k), -7.0, dtype=torch.float32, device=DEV)
        h.combine_ex(dev(q), out, y_scales=dev(s), recv_topk_weights=dev(rw), combined_topk_weights=cw)
        ref_out, ref_cw = oracle.combine_ex(R, E, k, idx, q, y_scales=s, recv_topk_weights=rw)
        frac = assert_bf16_close(host_bits(out), ref_out, "e4m3 combine")
        assert frac == 1.0
        assert np.array_equal(cw.cpu().numpy().view(np.uint32), ref_cw.view(np.uint32)), "combined_topk_weights"
        # without the weights' reduction, then with scales that are only
        # 4-byte aligned: the same values
        out2 = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
        h.combine_ex(dev(q), out2, y_scales=dev(s))
        assert np.array_equal(host_bits(out2), ref_out), "e4m3 combine without weights"
        s_buf = torch.empty(s.size + 1, dtype=torch.float32, device=DEV)
        s_off = s_buf[1:].view(P, H // 128)
        s_off.copy_(dev(s))
        out3 = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
        h.combine_ex(dev(q), out3, y_scales=s_off)
        assert np.array_equal(host_bits(out3), ref_out), "e4m3 combine, 4-byte aligned scales"
    # bf16 y through the general entry point equals the plain combine
    y = wl.normal_bf16(g, (P, H))
    out = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    h.combine_ex(dev(y), out)
    assert np.array_equal(host_bits(out), oracle.combine(R, E, k, idx, y))
    assert h.get_device_status() == ep.EP_OK
    h.close()


def test_combined_weights_undo_dispatch():
    """combine(recv_topk_weights of a dispatch) gives back the weights."""
    R, E, k, H, tpr = 8, 64, 8, 256, 40
    idx, w, x = _inputs(R, E, k, H, tpr, seed=90, dup=0.2)
    h, L, ref, _ = normal_path(R, E, k, H, idx, w, x, fp8=False)
    P = int(L["rank_offset"][-1])
    T = idx.shape[0]
    got = run_dispatch(h, dev(x), dev(w), False, P)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    cw = torch.empty((T, k), dtype=torch.float32, device=DEV)
    h.combine_ex(got["recv_x"], out, recv_topk_weights=got["recv_topk_weights"], combined_topk_weights=cw)
    assert np.array_equal(cw.cpu().numpy(), np.where(idx >= 0, w, np.float32(0)))
    h.close()


def test_combine_ex_argument_errors():
    R, E, k, H, tpr = 4, 16, 2, 256, 8
    idx, w, x = _inputs(R, E, k, H, tpr, seed=91)
    h, L, _, _ = normal_path(R, E, k, H, idx, w, x, fp8=False)
    P = int(L["rank_offset"][-1])
    T = idx.shape[0]
    out = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    y8 = torch.zeros((P, H), dtype=torch.uint8, device=DEV)
    rw = torch.zeros((P, k), dtype=torch.float32, device=DEV)
    L_ = ep.lib()
    # e4m3 rows without scales; weights in without weights out
    assert L_.ep_combine_ex(h.ptr, ep.EP_FP8_E4M3, y8.data_ptr(), None, P, None, out.data_ptr(), None, 0,
                            None) == ep.EP_ERR_INVALID_ARG
    assert L_.ep_combine_ex(h.ptr, ep.EP_BF16, y8.data_ptr(), None, P, rw.data_ptr(), out.data_ptr(), None, 0,
                            None) == ep.EP_ERR_INVALID_ARG
    assert L_.ep_combine_ex(h.ptr, 7, y8.data_ptr(), None, P, None, out.data_ptr(), None, 0,
                            None) == ep.EP_ERR_INVALID_ARG
    h.close()


@pytest.mark.parametrize("num_sms", [1, 3])
def test_combines_with_fewer_warps_than_parts(num_sms):
    """20 480 channels = 20 work items per token against 16 (bf16, 1 SM), 24
    (e4m3, 1 SM) or 48 warps: every warp steps its (token, part) by a whole
    number of tokens plus a remainder of parts, with the carry taken; every
    combine still equals the oracle."""
    R, E, k, H, tpr = 4, 16, 4, 20480, 16
    idx, w, x = _inputs(R, E, k, H, tpr, seed=300 + num_sms)
    T = idx.shape[0]
    L = oracle.layout(R, E, k, idx)
    P = int(L["rank_offset"][-1])
    y = wl.normal_bf16(wl.rng(301), (P, H))
    h, _, ref, frac = normal_path(R, E, k, H, idx, w, x, fp8=True, y=y, num_sms=num_sms)
    assert frac == 1.0
    rw = (wl.rng(302).random((P, k)) - 0.5).astype(np.float32)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    cw = torch.empty((T, k), dtype=torch.float32, device=DEV)
    h.combine_ex(dev(ref["recv_x"][:P]), out, y_scales=dev(ref["recv_scales"][:P]), recv_topk_weights=dev(rw),
                 combined_topk_weights=cw, num_sms=num_sms)
    ref_out, ref_cw = oracle.combine_ex(R, E, k, idx, ref["recv_x"][:P], y_scales=ref["recv_scales"][:P],
                                        recv_topk_weights=rw)
    assert np.array_equal(host_bits(out), ref_out)
    assert np.array_equal(cw.cpu().numpy().view(np.uint32), ref_cw.view(np.uint32))
    _, _, lfrac = ll_path(R, E, k, H, idx, w, x, fp8=False, y_seed=303, num_sms=num_sms, handle=h)
    assert lfrac == 1.0
    assert h.get_device_status() == ep.EP_OK
    h.close()


# ------------------------------------------------------------ int32 top-k ids

def _handle32(R, E, k, H, tpr):
    h = ep.Handle(R, E, k, H, tpr)
    h.set_topk_idx_bits(32)
    assert h.topk_idx_bits == 32
    return h


@pytest.mark.parametrize("case", CASES[:4], ids=[f"R{c[0]}E{c[1]}k{c[2]}H{c[3]}t{c[4]}" for c in CASES[:4]])
def test_int32_ids_every_routing_path(case):
    R, E, k, H, tpr = case
    idx, w, x = _inputs(R, E, k, H, tpr, seed=sum(case) + 5, dup=0.1)
    idx32 = idx.astype(np.int32)
    T = idx.shape[0]
    h = _handle32(R, E, k, H, tpr)
    # layout, then dispatch and combine on it
    L = oracle.layout(R, E, k, idx)
    ntpr = torch.full((R, R), -9, dtype=torch.int32, device=DEV)
    ntpe = torch.full((R, E), -9, dtype=torch.int32, device=DEV)
    itr = torch.zeros((T, R), dtype=torch.bool, device=DEV)
    h.get_dispatch_layout(dev(idx32), num_tokens_per_rank=ntpr, num_tokens_per_expert=ntpe, is_token_in_rank=itr)
    per_rank, per_expert, offset, _ = h.get_num_recv()
    assert np.array_equal(ntpr.cpu().numpy(), L["num_tokens_per_rank"])
    assert np.array_equal(ntpe.cpu().numpy(), L["num_tokens_per_expert"])
    assert np.array_equal(itr.cpu().numpy(), L["is_token_in_rank"])
    assert np.array_equal(offset, L["rank_offset"]) and np.array_equal(per_expert, L["num_recv_per_expert"])
    P = int(L["rank_offset"][-1])
    got = run_dispatch(h, dev(x), dev(w), True, P)
    ref, _ = oracle.dispatch(R, E, k, x, idx, w, fp8=True)
    assert np.array_equal(got["recv_x"].cpu().numpy(), ref["recv_x"][:P])
    assert np.array_equal(got["recv_topk_idx"].cpu().numpy(), ref["recv_topk_idx"][:P])
    # fused layout + dispatch
    recv = torch.empty((max(P, 1), H), dtype=torch.uint8, device=DEV)[:P]
    sc = torch.empty((max(P, 1), H // 128), dtype=torch.float32, device=DEV)[:P]
    src = torch.full((max(P, 1),), -7, dtype=torch.int32, device=DEV)[:P]
    h.layout_and_dispatch(dev(idx32), dev(x), dev(w), ep.EP_FP8_E4M3, recv, sc, recv_src_idx=src)
    assert np.array_equal(recv.cpu().numpy(), ref["recv_x"][:P])
    assert np.array_equal(src.cpu().numpy(), ref["recv_src_idx"][:P])
    # low latency
    M = h.M
    ll = torch.empty((E, M, H), dtype=torch.bfloat16, device=DEV)
    cnt = torch.full((E,), -7, dtype=torch.int32, device=DEV)
    info = torch.full((E, M), -7, dtype=torch.int32, device=DEV)
    h.low_latency_dispatch(dev(x), dev(idx32), ep.EP_BF16, ll, recv_src_info=info, recv_count=cnt)
    lref, _ = oracle.ll_dispatch(R, E, k, M, x, idx, fp8=False)
    count = cnt.cpu().numpy()
    assert np.array_equal(count, lref["recv_count"])
    for e in range(E):
        assert np.array_equal(info[e, :count[e]].cpu().numpy(), lref["recv_src_info"][e, :count[e]])
    assert h.get_device_status() == ep.EP_OK
    h.close()


def test_int32_ids_fused_v3_workload():
    """Full V3 shape with int32 ids through the fused layout + FP8 dispatch
    (a token's eight ids read as two 16-byte words): every output equals the
    oracle's, which routes the same ids as int64."""
    w_ = wl.WORKLOADS["v3_ep8"]
    x, idx, wts = wl.make_inputs(w_)
    R, E, k, H = w_.R, w_.E, w_.k, w_.H
    h = _handle32(R, E, k, H, w_.tokens_per_rank)
    ref, _ = oracle.dispatch(R, E, k, x, idx, wts, fp8=True)
    L = oracle.layout(R, E, k, idx)
    P = int(L["rank_offset"][-1])
    recv = torch.empty((P, H), dtype=torch.uint8, device=DEV)
    sc = torch.empty((P, H // 128), dtype=torch.float32, device=DEV)
    src = torch.full((P,), -7, dtype=torch.int32, device=DEV)
    ridx = torch.full((P, k), -7, dtype=torch.int32, device=DEV)
    rw = torch.full((P, k), -7.0, dtype=torch.float32, device=DEV)
    h.layout_and_dispatch(dev(idx.astype(np.int32)), dev(x), dev(wts), ep.EP_FP8_E4M3, recv, sc, recv_src_idx=src,
                          recv_topk_idx=ridx, recv_topk_weights=rw)
    _, _, offset, _ = h.get_num_recv()
    assert np.array_equal(offset, L["rank_offset"])
    assert np.array_equal(recv.cpu().numpy(), ref["recv_x"][:P])
    assert np.array_equal(sc.cpu().numpy().view(np.uint32), ref["recv_scales"][:P].view(np.uint32))
    assert np.array_equal(src.cpu().numpy(), ref["recv_src_idx"][:P])
    assert np.array_equal(ridx.cpu().numpy(), ref["recv_topk_idx"][:P])
    assert np.array_equal(rw.cpu().numpy().view(np.uint32), ref["recv_topk_weights"][:P].view(np.uint32))
    assert h.get_device_status() == ep.EP_OK
    h.close()


def test_int32_ids_fused_k8_bad_id_latched():
    """An out-of-range int32 id among a token's eight (the 16-byte id loads)
    is latched and routed nowhere; the other ids route as the oracle does
    with that entry masked."""
    R, E, k, H, tpr = 8, 64, 8, 256, 16
    idx, w, x = _inputs(R, E, k, H, tpr, seed=23)
    bad = idx.astype(np.int32)
    bad[5, 3] = E
    h = _handle32(R, E, k, H, tpr)
    masked = idx.copy()
    masked[5, 3] = -1
    L = oracle.layout(R, E, k, masked)
    P = int(L["rank_offset"][-1])
    recv = torch.empty((max(P, 1), H), dtype=torch.uint8, device=DEV)[:P]
    sc = torch.empty((max(P, 1), H // 128), dtype=torch.float32, device=DEV)[:P]
    h.layout_and_dispatch(dev(bad), dev(x), dev(w), ep.EP_FP8_E4M3, recv, sc)
    assert h.get_device_status() == ep.EP_ERR_BAD_EXPERT
    _, _, offset, _ = h.get_num_recv()
    assert np.array_equal(offset, L["rank_offset"])
    ref, _ = oracle.dispatch(R, E, k, x, masked, w, fp8=True)
    assert np.array_equal(recv.cpu().numpy(), ref["recv_x"][:P])
    h.close()


def test_int32_ids_bad_id_latched_and_width_checked():
    R, E, k, H, tpr = 4, 16, 2, 128, 8
    idx, w, x = _inputs(R, E, k, H, tpr, seed=17)
    idx32 = idx.astype(np.int32)
    idx32[3, 1] = E   # out of range
    h = _handle32(R, E, k, H, tpr)
    h.get_dispatch_layout(dev(idx32))
    assert h.get_device_status() == ep.EP_ERR_BAD_EXPERT
    # an int64 table on an int32 handle is refused before any launch
    with pytest.raises(ValueError):
        h.get_dispatch_layout(dev(idx))
    h.set_topk_idx_bits(64)
    idx[3, 1] = 1
    _, L, _, _ = normal_path(R, E, k, H, idx, w, x, fp8=False, handle=h)
    with pytest.raises(ep.EPError):
        h.set_topk_idx_bits(16)
    h.close()


def test_int32_ids_from_environment(monkeypatch):
    monkeypatch.setenv("EP_NUM_TOPK_IDX_BITS", "32")
    h = ep.Handle(4, 16, 2, 128, 8)
    assert h.topk_idx_bits == 32
    h.close()
    monkeypatch.setenv("EP_NUM_TOPK_IDX_BITS", "12")
    with pytest.raises(ep.EPError):
        ep.Handle(4, 16, 2, 128, 8)
    monkeypatch.delenv("EP_NUM_TOPK_IDX_BITS")
    h = ep.Handle(4, 16, 2, 128, 8)
    assert h.topk_idx_bits == 64
    h.close()


def test_combine_ex_v3_workload():
    """Full V3 shape: the e4m3 rows of the fused dispatch combined back, with
    the weights' reduction, against the oracle."""
    w_ = wl.WORKLOADS["v3_ep8"]
    x, idx, wts = wl.make_inputs(w_)
    R, E, k, H, T = w_.R, w_.E, w_.k, w_.H, w_.T
    L = oracle.layout(R, E, k, idx)
    P = int(L["rank_offset"][-1])
    h = ep.Handle(R, E, k, H, w_.tokens_per_rank)
    recv = torch.empty((P, H), dtype=torch.uint8, device=DEV)
    sc = torch.empty((P, H // 128), dtype=torch.float32, device=DEV)
    rw = torch.empty((P, k), dtype=torch.float32, device=DEV)
    h.layout_and_dispatch(dev(idx), dev(x), dev(wts), ep.EP_FP8_E4M3, recv, sc, recv_topk_weights=rw)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    cw = torch.empty((T, k), dtype=torch.float32, device=DEV)
    h.combine_ex(recv, out, y_scales=sc, recv_topk_weights=rw, combined_topk_weights=cw)
    ref_out, ref_cw = oracle.combine_ex(R, E, k, idx, recv.cpu().numpy(), y_scales=sc.cpu().numpy(),
                                        recv_topk_weights=rw.cpu().numpy())
    assert assert_bf16_close(host_bits(out), ref_out, "e4m3 combine, V3 shape") == 1.0
    assert np.array_equal(cw.cpu().numpy().view(np.uint32), ref_cw.view(np.uint32))
    assert np.array_equal(cw.cpu().numpy(), np.where(idx >= 0, wts, np.float32(0)))
    # the same rows without the weights' reduction
    out2 = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    h.combine_ex(recv, out2, y_scales=sc)
    assert np.array_equal(host_bits(out2), ref_out)
    assert h.get_device_status() == ep.EP_OK
    h.close()


def test_e4m3_combine_tokens_without_destinations():
    """Tokens whose every entry is masked combine to +0 (no source enters the
    three-slab register ring), next to tokens with up to 16 sources (the ring
    wraps five times)."""
    R, E, k, H, tpr = 16, 64, 16, 1024, 10
    idx, w, x = _inputs(R, E, k, H, tpr, seed=91, mask=0.05)
    idx[::3] = -1
    h, L, ref, _ = normal_path(R, E, k, H, idx, w, x, fp8=True)
    T = idx.shape[0]
    out = torch.full((T, H), 7.0, dtype=torch.bfloat16, device=DEV)
    P = int(L["rank_offset"][-1])
    h.combine_ex(dev(ref["recv_x"][:P]), out, y_scales=dev(ref["recv_scales"][:P]))
    ref_out, _ = oracle.combine_ex(R, E, k, idx, ref["recv_x"][:P], y_scales=ref["recv_scales"][:P])
    got = host_bits(out)
    assert np.array_equal(got, ref_out)
    assert not got[::3].any()
    assert h.get_device_status() == ep.EP_OK
    h.close()
