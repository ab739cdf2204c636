"""The allocation-free layout entry point (ep_get_dispatch_layout_noalloc).

Some callers cannot call cudaMalloc: serving runtimes that hand all device
memory to their own allocator up front, or plugin hosts that call in per
request with nowhere to keep a handle (creating one allocates).  This entry
point takes only caller buffers and keeps its scan state in a fixed array in
the library.  The tests check, on two calls in a row with different shapes
(so the shared array is reused and must be cleared between them):

* every output against the CPU oracle's layout, bit for bit: the counts,
  is_token_in_rank, rank_offset, and each token's (rank, row) list against
  the oracle's per-(token, rank) rows;
* every output against the handle-based ep_get_dispatch_layout, bit for bit,
  and that the destinations name the rows the handle's dispatch fills;
* that repeated calls leave the device's free memory (cudaMemGetInfo) and
  PyTorch's allocator unchanged after the first call's one-time set-up.

Collected last on purpose (file name), and self-contained: it passes alone in
a fresh process and after the rest of the suite.
"""
import numpy as np
import pytest
import torch

import oracle
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


def _outputs(R, E, k, T):
    kmax = min(k, R)
    return dict(
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


def _layout_noalloc(R, E, k, tpr, idx_d):
    out = _outputs(R, E, k, R * tpr)
    ep.ep_get_dispatch_layout_noalloc(R, E, k, idx_d, **out)
    return out


def _oracle_token_dest(slot, kmax):
    """(rank, row-in-rank) of every token's destinations, ascending rank,
    padded with (-1, -1): restated from the oracle's per-(token, rank) rows."""
    T, R = slot.shape
    dest = np.full((T, kmax, 2), -1, np.int32)
    for t in range(T):
        ranks = np.nonzero(slot[t] >= 0)[0]
        dest[t, : len(ranks), 0] = ranks
        dest[t, : len(ranks), 1] = slot[t, ranks]
    return dest


def test_noalloc_layout_matches_oracle_and_handle_layout_on_two_calls():
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
        torch.cuda.synchronize()
        assert int(got["device_status"].item()) == ep.EP_OK

        # against the oracle, bit for bit
        L = oracle.layout(R, E, k, idx)
        assert np.array_equal(got["num_tokens_per_rank"].cpu().numpy(), L["num_tokens_per_rank"])
        assert np.array_equal(got["num_tokens_per_expert"].cpu().numpy(), L["num_tokens_per_expert"])
        assert np.array_equal(got["is_token_in_rank"].cpu().numpy().astype(np.uint8), L["is_token_in_rank"])
        assert np.array_equal(got["num_recv_tokens_per_rank"].cpu().numpy(), L["num_recv_per_rank"])
        assert np.array_equal(got["num_recv_tokens_per_expert"].cpu().numpy(), L["num_recv_per_expert"])
        assert np.array_equal(got["rank_offset"].cpu().numpy(), L["rank_offset"])
        assert np.array_equal(got["token_dest"].cpu().numpy(), _oracle_token_dest(L["slot"], min(k, R)))
        assert np.array_equal(got["topk_idx32"].cpu().numpy(), idx.astype(np.int32))

        # against the handle-based layout, bit for bit
        h, ntpr, ntpe, itr, per_rank, per_expert, offset = _layout_via_handle(R, E, k, tpr, idx_d)
        torch.cuda.synchronize()
        assert torch.equal(got["num_tokens_per_rank"], ntpr)
        assert torch.equal(got["num_tokens_per_expert"], ntpe)
        assert torch.equal(got["is_token_in_rank"], itr)
        assert np.array_equal(got["num_recv_tokens_per_rank"].cpu().numpy(), per_rank)
        assert np.array_equal(got["num_recv_tokens_per_expert"].cpu().numpy(), per_expert)
        assert np.array_equal(got["rank_offset"].cpu().numpy(), offset)

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
        assert h.get_device_status() == ep.EP_OK
        h.close()


def test_noalloc_layout_allocates_nothing_on_repeated_calls():
    """After the first call on the device (its one-time set-up), further calls
    change neither the device's free memory nor PyTorch's allocator."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    R, E, k, tpr = 8, 256, 8, 1024
    T = R * tpr
    g = wl.rng(13)
    idx, _ = wl.route_uniform(g, T, E, k)
    idx_d = torch.from_numpy(idx).cuda()
    out = _outputs(R, E, k, T)
    ep.ep_get_dispatch_layout_noalloc(R, E, k, idx_d, **out)  # set-up call
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    torch_bytes0 = torch.cuda.memory_allocated()
    for _ in range(5):
        ep.ep_get_dispatch_layout_noalloc(R, E, k, idx_d, **out)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"device free memory changed by {free0 - free1} bytes"
    assert torch.cuda.memory_allocated() == torch_bytes0
    assert int(out["device_status"].item()) == ep.EP_OK
    L = oracle.layout(R, E, k, idx)
    assert np.array_equal(out["rank_offset"].cpu().numpy(), L["rank_offset"])


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


def test_noalloc_layout_wrapper_checks_the_id_table_shape():
    """A topk_idx narrower than num_topk columns is refused before the call
    (the kernel would read T*k ids)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    R, E, k, T = 4, 16, 4, 64
    out = _outputs(R, E, k, T)
    narrow = torch.zeros((T, k - 1), dtype=torch.int64, device="cuda")
    with pytest.raises(ValueError):
        ep.ep_get_dispatch_layout_noalloc(R, E, k, narrow, **out)
