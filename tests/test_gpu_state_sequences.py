"""GPU checks of the state the row-moving kernels share across launches on
one handle: the row-claim counter, the finished-block counter, the grid
barrier's generation and the per-block "published" words.  Every kernel
leaves them ready for the next; these tests interleave every path -- fused
rank-major, low-latency and expert-major dispatch (with and without the grid
barrier), the cached-handle scatter, the combines -- many times on one
handle, eagerly and as CUDA-graph replays, and check every result against
the oracle each time.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_get_03_gb300 import ep
from combine_ep_get_03_gb300 import workloads as wl
from harness import DEV, dev, host_bits

pytestmark = pytest.mark.gpu


def _inputs(R, E, k, H, T, seed):
    g = wl.rng(seed)
    idx, w = wl.route_uniform(g, T, E, k)
    idx = wl.mask_entries(g, idx, 0.02)
    x = wl.normal_bf16(g, (T, H))
    return idx, w, x


class Paths:
    """Every path on one handle, each returning its outputs as numpy."""

    def __init__(self, h, R, E, k, H, idx, w, x, align=16, num_sms=0):
        self.h, self.R, self.E, self.k, self.H, self.align, self.n = h, R, E, k, H, align, num_sms
        self.idx, self.w, self.x = idx, w, x
        self.T = idx.shape[0]
        self.idx_d, self.w_d, self.x_d = dev(idx), dev(w), dev(x)
        self.L = oracle.layout(R, E, k, idx)
        self.P = int(self.L["rank_offset"][-1])
        em = oracle.em_layout(R, E, k, idx, align)
        self.Q = int(em["expert_offset"][-1])
        G = H // 128
        self.recv = torch.empty((self.P, H), dtype=torch.uint8, device=DEV)
        self.sc = torch.empty((self.P, G), dtype=torch.float32, device=DEV)
        self.recv_bf = torch.empty((self.P, H), dtype=torch.bfloat16, device=DEV)
        self.y = dev(wl.normal_bf16(wl.rng(5), (self.P, H)))
        self.out = torch.empty((self.T, H), dtype=torch.bfloat16, device=DEV)
        self.ll = torch.empty((E, h.M, H), dtype=torch.uint8, device=DEV)
        self.ll_sc = torch.empty((E, h.M, G), dtype=torch.float32, device=DEV)
        self.cnt = torch.empty(E, dtype=torch.int32, device=DEV)
        self.em = torch.empty((self.Q, H), dtype=torch.uint8, device=DEV)
        self.em_sc = torch.empty((G, (self.Q + 3) // 4 * 4), dtype=torch.float32, device=DEV)
        self.em_src = torch.empty(self.Q, dtype=torch.int32, device=DEV)
        self.ref = dict(
            disp=oracle.dispatch(R, E, k, x, idx, w, fp8=True)[0],
            comb=oracle.combine(R, E, k, idx, host_bits(self.y)),
            ll=oracle.ll_dispatch(R, E, k, h.M, x, idx, fp8=True)[0],
            em=oracle.em_dispatch(R, E, k, x, idx, w, fp8=True, align=align)[0],
        )

    def run(self, name):
        h = self.h
        if name == "fused":
            h.layout_and_dispatch(self.idx_d, self.x_d, self.w_d, ep.EP_FP8_E4M3, self.recv, self.sc, num_sms=self.n)
        elif name == "scatter":
            h.dispatch(self.x_d, None, ep.EP_FP8_E4M3, self.recv, self.sc, num_sms=self.n)
        elif name == "combine":
            h.combine(self.y, self.out, num_sms=self.n)
        elif name == "ll":
            h.low_latency_dispatch(self.x_d, self.idx_d, ep.EP_FP8_E4M3, self.ll, self.ll_sc, recv_count=self.cnt,
                                   num_sms=self.n)
        elif name == "em":
            h.em_layout_and_dispatch(self.idx_d, self.x_d, self.w_d, ep.EP_FP8_E4M3, self.align, self.em, self.em_sc,
                                     recv_src_idx=self.em_src, num_sms=self.n)

    def check(self, name):
        r = self.ref
        if name in ("fused", "scatter"):
            assert np.array_equal(self.recv.cpu().numpy(), r["disp"]["recv_x"]), name
            assert np.array_equal(self.sc.cpu().numpy(), r["disp"]["recv_scales"]), name
        elif name == "combine":
            assert np.array_equal(host_bits(self.out), r["comb"]), name
        elif name == "ll":
            c = self.cnt.cpu().numpy()
            assert np.array_equal(c, r["ll"]["recv_count"]), name
            flat = np.concatenate([e * self.h.M + np.arange(n) for e, n in enumerate(c)]).astype(np.int64)
            got = self.ll.view(-1, self.H)[torch.from_numpy(flat).to(DEV)].cpu().numpy()
            assert np.array_equal(got, r["ll"]["recv_x"].reshape(-1, self.H)[flat]), name
        elif name == "em":
            src = self.em_src.cpu().numpy()
            assert np.array_equal(src, r["em"]["recv_src_idx"]), name
            real = src >= 0
            assert np.array_equal(self.em.cpu().numpy()[real], r["em"]["recv_x"][real]), name


SEQ = ["fused", "combine", "ll", "em", "scatter", "ll", "fused", "em", "em", "ll", "combine", "scatter", "fused"]


@pytest.mark.parametrize("T,R,E,k,H", [(256, 8, 64, 8, 512),     # small: per-entry paths without the grid barrier
                                       (4096, 8, 64, 8, 256)])   # 32768 entries: with the grid barrier
def test_interleaved_paths_on_one_handle(T, R, E, k, H):
    idx, w, x = _inputs(R, E, k, H, T, seed=T + R)
    h = ep.Handle(R, E, k, H, T // R)
    p = Paths(h, R, E, k, H, idx, w, x)
    for rep in range(3):
        for name in SEQ:
            p.run(name)
            p.check(name)
    assert h.get_device_status() == ep.EP_OK
    h.close()


@pytest.mark.parametrize("num_sms", [0, 9])
def test_interleaved_paths_as_graph_replays(num_sms):
    """The whole sequence captured once and replayed: every replay leaves the
    control words as the next kernel expects them."""
    T, R, E, k, H = 1024, 8, 64, 8, 512
    idx, w, x = _inputs(R, E, k, H, T, seed=33 + num_sms)
    h = ep.Handle(R, E, k, H, T // R)
    p = Paths(h, R, E, k, H, idx, w, x, num_sms=num_sms)
    seq = ["fused", "ll", "em", "scatter"]
    for name in seq:  # eager once: the layout must exist before the capture
        p.run(name)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for name in seq:
                p.run(name)
    torch.cuda.current_stream().wait_stream(s)
    for rep in range(5):
        p.recv.zero_()
        p.em.zero_()
        p.cnt.fill_(-1)
        g.replay()
        torch.cuda.synchronize()
        for name in seq:
            p.check(name)
    assert h.get_device_status() == ep.EP_OK
    h.close()


def test_a_smaller_handle_created_later_leaves_the_larger_one_working():
    """Kernels whose shared memory grows with R + E (the R > 64 layout, the
    low-latency routing fallback) keep working on a handle after a smaller
    handle is created: the per-kernel shared-memory limit does not follow the
    last handle's shape."""
    from harness import check_layout, ll_path

    R, k, H, tpr = 128, 8, 128, 8
    T = R * tpr
    big = ep.Handle(R, 1024, k, H, tpr)      # layout ~96 KB, low-latency routing ~91 KB of shared memory
    small = ep.Handle(R, 128, k, H, tpr)     # ~60 KB and ~55 KB
    for E, h in ((1024, big), (128, small), (1024, big)):
        g = wl.rng(40 + E)
        idx, w = wl.route_uniform(g, T, E, k)
        x = wl.normal_bf16(g, (T, H))
        check_layout(h, idx)
        # one SM: too many (token, k) entries for the fused kernel, so the
        # routing runs in the separate low-latency routing kernel
        ll_path(R, E, k, H, idx, w, x, fp8=True, num_sms=1, handle=h)
        assert h.get_device_status() == ep.EP_OK
    small.close()
    big.close()
