"""Pins for the oracle's general combine (an e4m3 input, the reduction of
the receive-side top-k weights) and for the expert-major ("GEMM") layout,
its dispatch and its combine.

As in the routing pins, each check stands apart from the oracle's loops:
hand-worked values (tests/golden/tiny_hand_worked.json), a brute-force
restatement by sorting, closed forms made exact by power-of-two scales or
identity experts, an exact-arithmetic bound, and an adjoint identity.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from combine_ep_get_03_gb300 import workloads as wl


def _hand(golden_dir):
    with open(os.path.join(golden_dir, "tiny_hand_worked.json")) as f:
        return json.load(f)


def _routing(T, R, E, k, seed, mask_frac=0.0, dup_frac=0.0):
    g = wl.rng(seed)
    idx, w = wl.route_uniform(g, T, E, k)
    if mask_frac:
        idx = wl.mask_entries(g, idx, mask_frac)
    if dup_frac:
        sel = g.random(T) < dup_frac
        idx[sel, k - 1] = idx[sel, 0]
    return idx, w


def _f32(bits):
    return wl.bf16_bits_to_f32(bits)


def _bf16(vals):
    return wl.f32_to_bf16_bits(np.asarray(vals, np.float32))


def _e4m3_decode(codes):
    """e4m3 bytes -> float64 through torch's float8_e4m3fn (a library routine)."""
    t = torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


# ------------------------------------------------- combine: top-k weights

def test_combine_weights_order_hand_worked(golden_dir):
    """The weights of one column are summed in ascending rank order: only that
    order keeps 2^-30."""
    h = _hand(golden_dir)
    c = h["combine_order"]
    R, E, k, H = c["R"], c["E"], c["k"], 128
    idx = np.array(c["topk_idx"], np.int64)
    y = _bf16(np.zeros((3, H)))
    rw = np.repeat(np.array(c["y_row_value"], np.float32)[:, None], k, 1)
    _, cw = oracle.combine_ex(R, E, k, idx, y, recv_topk_weights=rw)
    assert np.array_equal(cw, np.repeat(np.array(c["out_value"], np.float32)[:, None], k, 1))
    assert not np.signbit(cw).any()


@pytest.mark.parametrize("R,E,k,dup", [(4, 16, 2, 0.0), (8, 64, 8, 0.2), (64, 256, 8, 0.0)])
def test_combine_weights_undo_dispatch(R, E, k, dup):
    """Dispatch puts w[t][j] on the one rank that owns expert j and 0 on the
    others; summing the rows back gives w[t][j] exactly (0 where masked)."""
    T, H = R * 6, 128
    idx, w = _routing(T, R, E, k, seed=R + k, mask_frac=0.05, dup_frac=dup)
    x = wl.normal_bf16(wl.rng(R), (T, H))
    d, _ = oracle.dispatch(R, E, k, x, idx, w, fp8=False)
    _, cw = oracle.combine_ex(R, E, k, idx, d["recv_x"], recv_topk_weights=d["recv_topk_weights"])
    assert np.array_equal(cw, np.where(idx >= 0, w, np.float32(0)))


# ---------------------------------------------------- combine: e4m3 input

def _pow2_scaled_tokens(T, H, seed):
    """bf16 rows whose 128-channel group g of token t has |max| = 448 * 2^m
    with m = (t + 3 g) % 7 - 3, so that the group's scale is exactly 2^m."""
    g = wl.rng(seed)
    x = _f32(wl.normal_bf16(g, (T, H))).copy()
    for t in range(T):
        for gi in range(H // 128):
            m = (t + 3 * gi) % 7 - 3
            blk = x[t, gi * 128:(gi + 1) * 128]
            blk *= np.float32(100.0 * 2.0 ** m) / np.abs(blk).max()   # |values| < 448 * 2^m
            blk[g.integers(128)] = np.float32(448.0 * 2.0 ** m) * (1 if g.random() < 0.5 else -1)
    return _bf16(x)


@pytest.mark.parametrize("R,E,k", [(4, 16, 2), (8, 64, 8)])
def test_fp8_combine_power_of_two_scales_closed_form(R, E, k):
    """With every group scale a power of two, decode(q) * scale is exact and
    n copies of it add exactly: out[t] = bf16(n_t * decode(q[t]) * 2^m)."""
    T, H = R * 8, 384
    idx, w = _routing(T, R, E, k, seed=40 + R, mask_frac=0.05)
    x = _pow2_scaled_tokens(T, H, seed=41 + R)
    d, _ = oracle.dispatch(R, E, k, x, idx, w, fp8=True)
    src = d["recv_src_idx"]
    m = np.array([[(t + 3 * gi) % 7 - 3 for gi in range(H // 128)] for t in range(T)])
    assert np.array_equal(d["recv_scales"].astype(np.float64), np.exp2(m[src]))
    out, _ = oracle.combine_ex(R, E, k, idx, d["recv_x"], y_scales=d["recv_scales"])
    n = oracle.layout(R, E, k, idx)["is_token_in_rank"].sum(1)
    q_tok = np.zeros((T, H), np.uint8)
    q_tok[src] = d["recv_x"]
    exact = _e4m3_decode(q_tok) * np.repeat(np.exp2(m), 128, 1) * n[:, None]
    exact = exact + 0.0                              # the sum starts from +0: -0 codes give +0
    expect = _bf16(exact.astype(np.float32))        # exact in fp32: at most 7 significant bits
    assert np.array_equal(out, expect)


def test_fp8_combine_general_within_bound():
    """Random e4m3 rows and scales: |out - exact| <= 1/2 bf16 ulp(out) +
    n * 2^-23 * sum |decode * scale| against the float64 sum (each product
    rounds once, each of the n - 1 adds once)."""
    T, R, E, k, H = 128, 8, 64, 8, 256
    idx, w = _routing(T, R, E, k, seed=55, mask_frac=0.02)
    L = oracle.layout(R, E, k, idx)
    P = int(L["rank_offset"][-1])
    g = wl.rng(56)
    q = g.integers(0, 256, (P, H), dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x00                  # no NaN codes
    sc = (g.random((P, H // 128)) * 4 + 0.01).astype(np.float32)
    out = _f32(oracle.combine_ex(R, E, k, idx, q, y_scales=sc)[0]).astype(np.float64)
    v = _e4m3_decode(q) * np.repeat(sc.astype(np.float64), 128, 1)
    exact = np.zeros((T, H))
    absum = np.zeros((T, H))
    for t in range(T):
        for r in range(R):
            if L["slot"][t, r] >= 0:
                row = L["rank_offset"][r] + L["slot"][t, r]
                exact[t] += v[row]
                absum[t] += np.abs(v[row])
    n = L["is_token_in_rank"].sum(1)[:, None]
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(out), 1e-30))) - 7)
    assert np.all(np.abs(out - exact) <= 0.5 * ulp + n * 2.0 ** -23 * absum + 1e-30)


# ------------------------------------------------------ expert-major layout

def test_em_layout_hand_worked(golden_dir):
    h = _hand(golden_dir)
    em = h["expert_major"]
    R, E, k = h["R"], h["E"], h["k"]
    idx = np.array(h["topk_idx"], np.int64)
    for align in (1, 4):
        L = oracle.em_layout(R, E, k, idx, align)
        assert L["num_recv_per_expert"].tolist() == em["num_recv_per_expert"]
        assert L["expert_offset"].tolist() == em[f"align{align}_expert_offset"]
        assert L["row"].tolist() == em[f"align{align}_row"]
    H = 128
    x = _bf16(np.arange(h["T"], dtype=np.float32)[:, None] + np.zeros((1, H), np.float32))
    w = np.array(h["topk_weights"], np.float32)
    d, st = oracle.em_dispatch(R, E, k, x, idx, w, fp8=False, align=4)
    assert st == oracle.OK
    assert d["recv_src_idx"].tolist() == em["align4_recv_src_idx"]
    assert d["recv_weights"].tolist() == em["align4_recv_weights"]
    for row, t in enumerate(em["align4_recv_src_idx"]):
        assert np.all(_f32(d["recv_x"][row]) == (t if t >= 0 else 0))   # padding rows untouched


def _sorted_entries(idx, E, align):
    """Expert-major rows by brute force: sort the unmasked (expert, token,
    k-index) triples; offsets from numpy bincount / cumsum."""
    T, k = idx.shape
    t, j = np.nonzero(idx >= 0)
    e = idx[t, j]
    order = np.lexsort((j, t, e))
    counts = np.bincount(e, minlength=E) if len(e) else np.zeros(E, np.int64)
    padded = -(-counts // align) * align
    offset = np.concatenate([[0], np.cumsum(padded)])
    row = np.full((T, k), -1)
    first = np.concatenate([[0], np.cumsum(counts)])
    for pos, i in enumerate(order):
        row[t[i], j[i]] = offset[e[i]] + pos - first[e[i]]
    return counts, offset, row


@pytest.mark.parametrize("T,R,E,k,mask,dup,align", [(64, 4, 16, 2, 0.0, 0.0, 1), (96, 8, 64, 6, 0.05, 0.1, 4),
                                                     (120, 3, 12, 4, 0.2, 0.3, 128), (32, 32, 32, 8, 0.01, 0.0, 8),
                                                     (0, 4, 8, 2, 0.0, 0.0, 4)])
def test_em_layout_vs_sorted_entries(T, R, E, k, mask, dup, align):
    idx, _ = _routing(T, R, E, k, seed=T + E + align, mask_frac=mask, dup_frac=dup)
    idx = idx.reshape(T, k)
    L = oracle.em_layout(R, E, k, idx, align)
    counts, offset, row = _sorted_entries(idx, E, align)
    assert L["num_recv_per_expert"].tolist() == counts.tolist()
    assert L["expert_offset"].tolist() == offset.tolist()
    assert np.array_equal(L["row"], row)
    assert np.all(L["expert_offset"] % align == 0)


@pytest.mark.parametrize("fp8", [False, True])
def test_em_dispatch_rows_and_padding(fp8):
    T, R, E, k, H, align = 96, 4, 32, 4, 256, 8
    idx, w = _routing(T, R, E, k, seed=15, mask_frac=0.05, dup_frac=0.1)
    x = wl.normal_bf16(wl.rng(16), (T, H))
    d, st = oracle.em_dispatch(R, E, k, x, idx, w, fp8=fp8, align=align)
    assert st == oracle.OK
    L = oracle.em_layout(R, E, k, idx, align)
    rows = int(L["expert_offset"][-1])
    seen = np.zeros(rows, bool)
    for t in range(T):
        q, s = oracle.quantize_row(x[t]) if fp8 else (None, None)
        for j in range(k):
            r_ = L["row"][t, j]
            if r_ < 0:
                continue
            assert not seen[r_]
            seen[r_] = True
            e = idx[t, j]
            assert L["expert_offset"][e] <= r_ < L["expert_offset"][e] + L["num_recv_per_expert"][e]
            assert d["recv_src_idx"][r_] == t and d["recv_weights"][r_] == w[t, j]
            if fp8:
                assert np.array_equal(d["recv_x"][r_], q)
                assert np.array_equal(d["recv_scales"][:, r_], s)      # group-major
            else:
                assert np.array_equal(d["recv_x"][r_], x[t])
    assert np.all(d["recv_src_idx"][~seen] == -1) and np.all(d["recv_weights"][~seen] == 0)
    assert np.all(d["recv_x"][~seen] == 0)
    if fp8:
        assert np.all(d["recv_scales"][:, :rows][:, ~seen] == -7.0)    # padding scales unwritten


def test_em_dispatch_capacity_skips_rows():
    T, R, E, k, H, align = 64, 4, 16, 2, 128, 4
    idx, w = _routing(T, R, E, k, seed=3)
    x = wl.normal_bf16(wl.rng(4), (T, H))
    full, st = oracle.em_dispatch(R, E, k, x, idx, w, fp8=False, align=align)
    rows = full["recv_x"].shape[0]
    part, st2 = oracle.em_dispatch(R, E, k, x, idx, w, fp8=False, align=align, capacity_rows=rows - 9)
    assert st == oracle.OK and st2 == oracle.CAPACITY
    assert np.array_equal(part["recv_x"], full["recv_x"][: rows - 9])
    assert np.array_equal(part["recv_src_idx"], full["recv_src_idx"][: rows - 9])


# ----------------------------------------------------- expert-major combine

def test_em_combine_order_hand_worked(golden_dir):
    c = _hand(golden_dir)["em_combine_order"]
    H = 128
    idx = np.array(c["topk_idx"], np.int64)
    y = _bf16(np.repeat(np.array(c["y_row_value"], np.float32)[:, None], H, 1))
    out = oracle.em_combine(c["R"], c["E"], c["k"], idx, 1, y)
    assert np.array_equal(_f32(out), np.repeat(np.array(c["out_value"], np.float32)[:, None], H, 1))
    assert not np.signbit(_f32(out[1:])).any()


@pytest.mark.parametrize("R,E,k,align", [(4, 16, 2, 1), (8, 64, 8, 16), (64, 256, 8, 4)])
def test_em_combine_identity_expert_closed_form(R, E, k, align):
    """y = the dispatched rows: out[t] = bf16(n_t * x[t]), n_t = the token's
    unmasked entries (n_t * x is exact in fp32, and so is every partial sum)."""
    T, H = R * 8, 256
    idx, w = _routing(T, R, E, k, seed=R + align, mask_frac=0.05, dup_frac=0.1)
    x = wl.normal_bf16(wl.rng(R + 1), (T, H))
    d, _ = oracle.em_dispatch(R, E, k, x, idx, w, fp8=False, align=align)
    out = oracle.em_combine(R, E, k, idx, align, d["recv_x"])
    n = (idx >= 0).sum(1).astype(np.float32)
    expect = wl.f32_to_bf16_bits(_f32(x) * n[:, None])
    expect[n == 0] = 0
    assert np.array_equal(out, expect)


def test_em_dispatch_combine_adjoint():
    """<em_dispatch(g), y> == <g, em_combine(y)> over the real rows, float64."""
    T, R, E, k, H, align = 96, 4, 32, 4, 128, 4
    idx, w = _routing(T, R, E, k, seed=97, mask_frac=0.03)
    g = wl.normal_bf16(wl.rng(98), (T, H), sigma=1e-2)
    d, _ = oracle.em_dispatch(R, E, k, g, idx, w, fp8=False, align=align)
    real = d["recv_src_idx"] >= 0
    y = wl.normal_bf16(wl.rng(99), (d["recv_x"].shape[0], H))
    y[~real] = _bf16(np.full(H, 1e3, np.float32))    # padding rows must not reach the output
    lhs = float((_f32(d["recv_x"][real]).astype(np.float64) * _f32(y[real]).astype(np.float64)).sum())
    comb = _f32(oracle.em_combine(R, E, k, idx, align, y)).astype(np.float64)
    rhs = float((_f32(g).astype(np.float64) * comb).sum())
    scale = float(np.abs(_f32(g)).astype(np.float64).sum() * np.abs(comb).max())
    assert abs(lhs - rhs) <= 2.0 ** -7 * scale
