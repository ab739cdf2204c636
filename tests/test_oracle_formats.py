"""Pins for the oracle's number formats (E4M3 encode/decode, bf16 rounding).

The oracle's encoders are written from the format definitions; here they are
checked against hand-encoded points (tests/golden/number_formats.json) and
against PyTorch's own float8_e4m3fn / bfloat16 conversions, an independent
library implementation of the same formats.
"""
import json
import os
import struct

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _golden(golden_dir):
    with open(os.path.join(golden_dir, "number_formats.json")) as f:
        return json.load(f)


def test_e4m3_hand_encoded_points(golden_dir):
    for p in _golden(golden_dir)["e4m3"]:
        assert oracle.float_to_e4m3(p["value"]) == p["code"], p


def test_bf16_hand_rounded_points(golden_dir):
    for p in _golden(golden_dir)["bf16"]:
        f = struct.unpack("<f", bytes.fromhex(p["value_hex_f32"])[::-1])[0]
        assert oracle.float_to_bf16(f) == int(p["bf16_hex"], 16), p


def test_e4m3_decode_all_codes_vs_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    got = np.array([oracle.e4m3_to_float(int(c)) for c in codes], np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert nan.sum() == 2  # 0x7f and 0xff
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))
    # magnitudes are strictly increasing over 0x00..0x7e
    assert np.all(np.diff(got[:127]) > 0)
    assert got[0x7E] == 448.0


def _torch_e4m3(v: np.ndarray) -> np.ndarray:
    return torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_encode_all_bf16_patterns_vs_torch():
    """Every bf16 bit pattern (as fp32) below the saturation point encodes as
    PyTorch's round-to-nearest-even float8_e4m3fn does."""
    bits = np.arange(65536, dtype=np.uint32) << 16
    v = bits.view(np.float32)
    keep = np.isfinite(v) & (np.abs(v) < 464.0)
    v = v[keep]
    got = oracle.float_to_e4m3_array(v)
    assert np.array_equal(got, _torch_e4m3(v))


def test_e4m3_encode_dense_fp32_sweep_vs_torch():
    """fp32 values with full 24-bit significands across every e4m3 binade,
    including the exact midpoints between neighbouring codes."""
    g = np.random.Generator(np.random.PCG64(7))
    exps = g.integers(-13, 9, 60000)
    mant = g.random(60000) + 1.0
    sign = np.where(g.random(60000) < 0.5, -1.0, 1.0)
    v = (sign * mant * np.exp2(exps)).astype(np.float32)
    codes = np.arange(0, 0x7F, dtype=np.uint8)
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    mids = ((vals[:-1].astype(np.float64) + vals[1:]) / 2).astype(np.float32)
    v = np.concatenate([v, mids, -mids, vals, -vals])
    v = v[np.abs(v) < 464.0]
    assert np.array_equal(oracle.float_to_e4m3_array(v), _torch_e4m3(v))


def test_e4m3_saturates():
    for f in (448.0001, 463.9, 464.0, 480.0, 1e6, 3.0e38, float("inf")):
        assert oracle.float_to_e4m3(f) == 0x7E
        assert oracle.float_to_e4m3(-f) == 0xFE


def test_bf16_rounding_vs_torch():
    g = np.random.Generator(np.random.PCG64(11))
    u = g.integers(0, 2**32, 200000, dtype=np.uint64).astype(np.uint32)
    # make a quarter of them exact ties and a quarter near ties
    u[::4] = (u[::4] & 0xFFFF0000) | 0x8000
    u[1::4] = (u[1::4] & 0xFFFF0000) | 0x7FFF
    v = u.view(np.float32)
    v = v[np.isfinite(v)]
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.float_to_bf16(float(x)) for x in v[:50000]], np.uint16)
    assert np.array_equal(got, ref[:50000])
