"""ep_get_buffer_size_hint (host only, no GPU): the rows it reports are the
most any routing can need -- reached by constructed worst-case routings,
never exceeded by random ones -- with the oracle's layouts as the measure."""
import numpy as np
import pytest

import oracle
from combine_ep_get_03_gb300 import build as cuda_build
from combine_ep_get_03_gb300 import workloads as wl


@pytest.fixture(scope="module")
def ep():
    cuda_build.build()
    from combine_ep_get_03_gb300 import ep as ep_mod
    return ep_mod


def _worst_rank_major(R, E, k, T):
    """Every token on min(k, R) distinct ranks."""
    El = E // R
    idx = np.full((T, k), -1, np.int64)
    for t in range(T):
        for j in range(k):
            idx[t, j] = ((t + j) % R) * El + (j // R) % El
    return idx


def _worst_expert_major(E, k, T, align, seed):
    """All entries unmasked and every expert count = 1 (mod align), so every
    group carries align - 1 padding rows."""
    n = T * k
    base = np.ones(E, np.int64)
    left = n - E
    assert left >= 0 and left % align == 0
    g = wl.rng(seed)
    extra = np.bincount(g.integers(0, E, left // align), minlength=E) * align
    ids = np.repeat(np.arange(E), base + extra)
    g.shuffle(ids)
    return ids.reshape(T, k)


@pytest.mark.parametrize("R,E,k,tpr", [(4, 16, 2, 10), (8, 64, 8, 16), (8, 256, 8, 12), (64, 256, 8, 2)])
def test_hint_rows_are_tight(ep, R, E, k, tpr):
    T = R * tpr
    rows, _ = ep.ep_get_buffer_size_hint(R, E, k, 256, tpr, ep.EP_BF16, ep.EP_LAYOUT_RANK_MAJOR)
    assert rows == T * min(k, R)
    assert oracle.layout(R, E, k, _worst_rank_major(R, E, k, T))["rank_offset"][-1] == rows
    for seed in range(3):
        idx, _ = wl.route_uniform(wl.rng(seed), T, E, k)
        assert oracle.layout(R, E, k, idx)["rank_offset"][-1] <= rows
    for align in (1, 4, 8):
        rows_em, _ = ep.ep_get_buffer_size_hint(R, E, k, 256, tpr, ep.EP_FP8_E4M3, ep.EP_LAYOUT_EXPERT_MAJOR, align)
        assert rows_em == T * k + E * (align - 1)
        if (T * k - E) >= 0 and (T * k - E) % align == 0:
            idx = _worst_expert_major(E, k, T, align, seed=align)
            assert oracle.em_layout(R, E, k, idx, align)["expert_offset"][-1] == rows_em
        idx, _ = wl.route_uniform(wl.rng(9), T, E, k)
        assert oracle.em_layout(R, E, k, idx, align)["expert_offset"][-1] <= rows_em
    rows_ll, _ = ep.ep_get_buffer_size_hint(R, E, k, 256, tpr, ep.EP_BF16, ep.EP_LAYOUT_LOW_LATENCY)
    assert rows_ll == E * T


def test_hint_bytes_match_the_buffers(ep):
    R, E, k, H, tpr = 8, 256, 8, 7168, 1024
    T, G = R * tpr, H // 128
    rows, b = ep.ep_get_buffer_size_hint(R, E, k, H, tpr, ep.EP_FP8_E4M3, ep.EP_LAYOUT_RANK_MAJOR)
    # recv_x e4m3 + scales + src_idx + topk idx + topk weights
    assert b == rows * H + rows * G * 4 + rows * 4 + rows * k * 4 + rows * k * 4
    rows, b = ep.ep_get_buffer_size_hint(R, E, k, H, tpr, ep.EP_BF16, ep.EP_LAYOUT_LOW_LATENCY)
    assert b == rows * 2 * H + rows * 4 + E * 4
    rows, b = ep.ep_get_buffer_size_hint(R, E, k, H, tpr, ep.EP_FP8_E4M3, ep.EP_LAYOUT_EXPERT_MAJOR, 128)
    ld = (rows + 3) // 4 * 4
    assert b == rows * H + G * ld * 4 + rows * 4 + rows * 4


def test_hint_rejects_bad_arguments(ep):
    with pytest.raises(ep.EPError):
        ep.ep_get_buffer_size_hint(8, 100, 8, 256, 4, ep.EP_BF16, ep.EP_LAYOUT_RANK_MAJOR)   # E % R != 0
    with pytest.raises(ep.EPError):
        ep.ep_get_buffer_size_hint(8, 64, 8, 200, 4, ep.EP_BF16, ep.EP_LAYOUT_RANK_MAJOR)    # H % 128 != 0
    with pytest.raises(ep.EPError):
        ep.ep_get_buffer_size_hint(8, 64, 8, 256, 4, ep.EP_BF16, ep.EP_LAYOUT_EXPERT_MAJOR, 0)
