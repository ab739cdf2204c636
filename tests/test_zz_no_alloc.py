"""The allocation-free layout entry point (ep_get_dispatch_layout_noalloc).

It serves callers that cannot call cudaMalloc (inside a stream capture, under
a runtime that owns all device memory, or without a place to keep a handle),
so it takes only caller buffers and keeps its scan state in a fixed array in
the library.  Two calls in a row, on different shapes so the shared array is
reused, must give exactly what the handle-based ep_get_dispatch_layout gives
(integer outputs: bit-exact), and its per-token destinations must name the
receive rows where the handle's dispatch put each token.

Collected last on purpose (file name), and self-contained: it passes alone in
a fresh process and after the rest of the suite.
"""
import numpy as np
import pytest
import torch

from combine_ep_get_03_gb300 import ep
from combine_ep_get_03_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

# (R, E, k, tokens per rank, seed): the V3 shape, then 64 ranks x 512 tokens
CASES = [(8, 256, 8, 1024, 11), (64, 256, 8, 512, 12)]


def _layout_via_handle(R, E, k, tpr, idx_d):
    T = R * tpr
    h = ep.Handle(R, E, k, 128, tpr)
    ntpr = torch.full((R, R), -9, dtype=torch.int32, device="cuda")
    ntpe = torch.full((R, E), -9, dtype=torch.int32, device="cuda")
    itr = torch.zeros((T, R), dtype=torch.bool, device="cuda")
    h.get_dispatch_layout(idx_d, num_tokens_per_rank=ntpr, num_tokens_per_expert=ntpe, is_token_in_rank=itr)
    per_rank, per_expert, offset, st = h.get_num_recv()
    assert st == ep.EP_OK
    return h, ntpr, ntpe, itr, per_rank, per_expert, offset


def _layout_noalloc(R, E, k, tpr, idx_d):
    T = R * tpr
    kmax = min(k, R)
    out = dict(
        num_tokens_per_rank=torch.full((R, R), -9, dtype=torch.int32, device="cuda"),
        num_tokens_per_expert=torch.full((R, E), -9, dtype=torch.int32, device="cuda"),
        is_token_in_rank=torch.zeros((T, R), dtype=torch.bool, device="cuda"),
        num_recv_tokens_per_rank=torch.full((R,), -9, dtype=torch.int32, device="cuda"),
        num_recv_tokens_per_expert=torch.full((E,), -9, dtype=torch.int32, device="cuda"),
        rank_offset=torch.full((R + 1,), -9, dtype=torch.int32, device="cuda"),
        token_dest=torch.full((T, kmax, 2), -9, dtype=torch.int32, device="cuda"),
        topk_idx32=torch.full((T, k), -9, dtype=torch.int32, device="cuda"),
        device_status=torch.zeros(1, dtype=torch.int32, device="cuda"),
    )
    ep.ep_get_dispatch_layout_noalloc(R, E, k, idx_d, **out)
    return out


def test_noalloc_layout_matches_handle_layout_on_two_calls():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    for R, E, k, tpr, seed in CASES:
        T = R * tpr
        g = wl.rng(seed)
        idx, _ = wl.route_uniform(g, T, E, k)
        idx = wl.mask_entries(g, idx, 0.01)
        idx_d = torch.from_numpy(idx).cuda()

        got = _layout_noalloc(R, E, k, tpr, idx_d)
        h, ntpr, ntpe, itr, per_rank, per_expert, offset = _layout_via_handle(R, E, k, tpr, idx_d)
        torch.cuda.synchronize()

        assert int(got["device_status"].item()) == ep.EP_OK
        assert torch.equal(got["num_tokens_per_rank"], ntpr)
        assert torch.equal(got["num_tokens_per_expert"], ntpe)
        assert torch.equal(got["is_token_in_rank"], itr)
        assert np.array_equal(got["num_recv_tokens_per_rank"].cpu().numpy(), per_rank)
        assert np.array_equal(got["num_recv_tokens_per_expert"].cpu().numpy(), per_expert)
        assert np.array_equal(got["rank_offset"].cpu().numpy(), offset)
        ids = idx.astype(np.int32)
        assert np.array_equal(got["topk_idx32"].cpu().numpy(), ids)

        # the destinations name the rows the handle's dispatch fills
        P = int(offset[-1])
        x = torch.zeros((T, 128), dtype=torch.bfloat16, device="cuda")
        recv = torch.empty((P, 128), dtype=torch.bfloat16, device="cuda")
        src = torch.full((P,), -1, dtype=torch.int32, device="cuda")
        h.dispatch(x, None, ep.EP_BF16, recv, recv_src_idx=src)
        dest = got["token_dest"].cpu().numpy()
        valid = dest[..., 0] >= 0
        rows = offset[dest[..., 0].clip(0)] + dest[..., 1]
        from_dest = np.full(P, -1, np.int64)
        tok = np.broadcast_to(np.arange(T)[:, None], valid.shape)
        from_dest[rows[valid]] = tok[valid]
        assert np.array_equal(from_dest, src.cpu().numpy())
        # ascending ranks, padding at the end
        r = np.where(valid, dest[..., 0], np.iinfo(np.int32).max)
        assert np.all((np.diff(r, axis=1) > 0) | ~valid[:, 1:])
        assert np.all(valid[:, :-1] | ~valid[:, 1:])
        assert h.get_device_status() == ep.EP_OK
        h.close()


def test_noalloc_layout_rejects_sizes_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    R, E, k, tpr = 1024, 4096, 8, 256  # 1024 * 2 chunks * 5120 columns > 131040 words
    idx_d = torch.zeros((R * tpr, k), dtype=torch.int64, device="cuda")
    dummy = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(ep.EPError) as e:
        ep.ep_get_dispatch_layout_noalloc(R, E, k, idx_d, torch.zeros(R, dtype=torch.int32, device="cuda"),
                                          torch.zeros(E, dtype=torch.int32, device="cuda"),
                                          torch.zeros(R + 1, dtype=torch.int32, device="cuda"),
                                          torch.zeros((R * tpr, k, 2), dtype=torch.int32, device="cuda"),
                                          torch.zeros((R * tpr, k), dtype=torch.int32, device="cuda"),
                                          device_status=dummy)
    assert e.value.status == ep.EP_ERR_INVALID_ARG
