"""Host-side arithmetic of the benchmark on CPU: the byte counts its metric
divides by, and the reading of the clock samples that decide whether a
measurement stands."""
import torch

import bench
from combine_ep_get_03_gb300 import workloads as wl


def test_logical_and_algorithmic_bytes_follow_their_definitions():
    """Logical bytes are rows moved x row payload (FP8 row: H bytes + H/128
    fp32 scales; BF16 row: 2H); algorithmic bytes count x read once per token
    and each receive row once."""
    w = wl.WORKLOADS["v3_ep8"]
    T, H, k, R = w.T, w.H, w.k, w.R
    P, n_ll = 43365, 65536
    s = bench.Sizes(w, P, n_ll)
    fp8_row = H + 4 * (H // 128)
    assert fp8_row == 7392
    assert s.logical["layout_dispatch_fp8"] == P * fp8_row
    assert s.logical["combine"] == s.logical["combine_bwd"] == s.logical["dispatch_bf16_bwd"] == P * 2 * H
    assert s.logical["ll_dispatch_fp8"] == n_ll * fp8_row
    assert s.logical["ll_combine"] == n_ll * 2 * H
    kmax = min(k, R)
    # combine: every receive row read once, every output row written once,
    # and the (rank, row) list of each token
    assert s.hbm["combine"] == P * 2 * H + T * 2 * H + 8 * T * kmax
    # backward dispatch: x-sized gradient read once, P rows written
    assert s.hbm["dispatch_bf16_bwd"] == T * 2 * H + P * 2 * H + 8 * T * kmax
    # low-latency combine: every unmasked entry's row, the weights and ids
    assert s.hbm["ll_combine"] == n_ll * 2 * H + T * 2 * H + 4 * T * k + 8 * T * k
    # the V3 figures quoted beside the bench line
    assert abs(s.hbm["combine"] - 739.6e6) < 0.1e6
    assert s.logical["combine"] == 43365 * 14336 == 621_680_640


def _sampler(lines):
    c = bench.ClockSampler(torch.device("cpu"))
    c.lines = lines
    return c


def test_clock_samples_give_median_max_and_active_reasons():
    lines = [
        "2070, 2070, 900.1, Not Active, Not Active, Not Active, Not Active",
        "2055, 2070, 1350.0, Not Active, Not Active, Not Active, Active",
        "2070, 2070, 1100.0, Not Active, Not Active, Not Active, Not Active",
        "not, a, sample",
    ]
    s = _sampler(lines).summary()
    assert s["sm_mhz"] == 2070.0
    assert s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]
    assert s["samples"] == 3


def test_clock_slowdowns_are_reported():
    lines = ["1500, 2070, 700.0, Active, Not Active, Active, Not Active"]
    s = _sampler(lines).summary()
    assert s["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    assert s["sm_mhz"] == 1500.0


def test_no_samples_is_not_a_clock_reading():
    s = _sampler([]).summary()
    assert s["sm_mhz"] is None and s["samples"] == 0


def test_reference_arm_rows_match_the_oracle_layout():
    """The reference arm's config reports the same receive rows as the GPU
    arm, whose rows come from the layout: check them against the oracle's."""
    import oracle
    from combine_ep_get_03_gb300 import workloads as wl

    for name in ("tiny_bf16", "v3_ep8"):
        w = wl.WORKLOADS[name]
        _, idx, _ = wl.make_inputs(w, rep=0)
        P, n_ll = bench.workload_rows(w)
        assert P == int(oracle.layout(w.R, w.E, w.k, idx)["rank_offset"][-1])
        has_ll = "ll_dispatch_fp8" in bench.OPS_OF.get(name, bench.OPS)
        assert n_ll == (int((idx >= 0).sum()) if has_ll else 0)
    cfg = bench.step_config(wl.WORKLOADS["v3_ep8"], 1, 2, 152, 1)
    assert {"workload", "dispatch", "combine", "recv_rows", "ll_rows", "num_sms", "parallelism"} <= set(cfg)


def test_cpu_model_and_cores_are_reported():
    assert bench.cpu_model()
    assert bench.host_cores() >= 1
