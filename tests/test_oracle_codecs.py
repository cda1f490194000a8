"""Pins of the oracle's number codecs and per-entry decode, against the formats' definitions
and library casts (torch CPU float8_e4m3fn / bfloat16), never against the oracle itself."""
import math
import struct

import numpy as np
import pytest
import torch


def torch_e4m3_value(code: int) -> float:
    return float(torch.tensor([code], dtype=torch.uint8).view(torch.float8_e4m3fn).float()[0])


def test_e4m3_decode_all_codes_match_torch(orc):
    vals = orc.e4m3_to_f64(np.arange(256))
    for c in range(256):
        ref = torch_e4m3_value(c)
        if math.isnan(ref):
            assert math.isnan(vals[c]), c
        else:
            assert vals[c] == ref, (c, vals[c], ref)


def test_e4m3_format_facts(orc):
    v = orc.e4m3_to_f64
    assert v([0x7E])[0] == 448.0                      # largest finite
    assert v([0x01])[0] == 2.0 ** -9                  # smallest subnormal
    assert v([0x08])[0] == 2.0 ** -6                  # smallest normal
    assert v([0x38])[0] == 1.0
    assert v([0x44])[0] == 3.0
    assert math.isnan(v([0x7F])[0]) and math.isnan(v([0xFF])[0])
    assert math.copysign(1.0, v([0x80])[0]) == -1.0 and v([0x80])[0] == 0.0
    # exactly two NaN codes, 254 finite ones, strictly increasing over 0x00..0x7E
    pos = v(np.arange(0x7F))
    assert np.all(np.diff(pos) > 0)


def _torch_encode(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.clip(x.astype(np.float32), -448.0, 448.0))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_encode_matches_torch_on_grid_ties_and_random(orc):
    grid = orc.e4m3_to_f64(np.arange(0x7F))
    mids = (grid[:-1] + grid[1:]) / 2
    xs = [grid, mids, np.nextafter(mids.astype(np.float32), np.float32(np.inf)),
          np.nextafter(mids.astype(np.float32), np.float32(-np.inf))]
    rng = np.random.default_rng(123)
    xs.append(rng.uniform(-600, 600, 3000))
    xs.append(rng.uniform(-0.02, 0.02, 3000))
    xs.append(np.array([0.0, 447.9, 448.0, 449.0, 464.0, 465.0, 1e9, -1e9, 2.0 ** -10, 2.0 ** -11,
                        3 * 2.0 ** -11]))
    x = np.concatenate([np.asarray(a, dtype=np.float64) for a in xs]).astype(np.float32)
    x = np.concatenate([x, -x])
    ours = orc.e4m3_from_f32(x)
    ref = _torch_encode(x)
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, [(float(x[i]), int(ours[i]), int(ref[i])) for i in bad[:10]]


def test_e4m3_encode_saturates_and_keeps_sign(orc):
    e = orc.e4m3_from_f32
    assert e([1e30])[0] == 0x7E and e([-1e30])[0] == 0xFE
    assert e([np.float32("-0.0")])[0] == 0x80
    assert e([np.nan])[0] == 0x7F


def test_bf16_codec_matches_torch(orc):
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.standard_normal(4000).astype(np.float32),
                        (rng.standard_normal(1000) * 1e30).astype(np.float32),
                        (rng.standard_normal(1000) * 1e-38).astype(np.float32)])
    # exact ties: bf16 value + half an ulp
    b = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    ulp_half = np.abs(b) * 2.0 ** -8
    x = np.concatenate([x, (b + ulp_half).astype(np.float32), (b - ulp_half).astype(np.float32)])
    ours = orc.bf16_from_f32(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = orc.bf16_to_f64(ref)
    assert np.array_equal(back, torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).double().numpy())


def test_decode_entry_formats(orc):
    rng = np.random.default_rng(5)
    # fp8_ds_mla: 512 e4m3 | 4 fp32 scales | 64 bf16
    rec = np.zeros(656, dtype=np.uint8)
    rec[:512] = rng.integers(0, 0x7F, 512)
    scales = np.array([0.5, 3.0, 0.0625, 7.25], dtype=np.float32)
    rec[512:528] = scales.view(np.uint8)
    rope = torch.randn(64).to(torch.bfloat16)
    rec[528:656] = rope.view(torch.int16).numpy().view(np.uint8)
    k = orc.decode_entry(orc.DS_MLA, rec)
    e = torch.from_numpy(rec[:512].copy()).view(torch.float8_e4m3fn).double().numpy()
    exp_nope = e * np.repeat(scales.astype(np.float64), 128)
    assert np.array_equal(k[:512], exp_nope)
    assert np.array_equal(k[512:], rope.double().numpy())
    # plain fp8: all 576 are e4m3 (no scale)
    ent = rng.integers(0, 0x7F, 576).astype(np.uint8)
    k = orc.decode_entry(orc.FP8, ent)
    assert np.array_equal(k, torch.from_numpy(ent).view(torch.float8_e4m3fn).double().numpy())
    # bf16: 576 little-endian bf16
    v = torch.randn(576).to(torch.bfloat16)
    k = orc.decode_entry(orc.BF16, v.view(torch.int16).numpy().view(np.uint8))
    assert np.array_equal(k, v.double().numpy())


def test_ds_tile_exponent_is_minimal_power_of_two(orc):
    rng = np.random.default_rng(9)
    amaxes = list(np.abs(rng.standard_normal(2000)) * 10.0 ** rng.uniform(-6, 6, 2000))
    amaxes += [448.0 * 2.0 ** k for k in range(-20, 10)]
    amaxes += [np.nextafter(448.0 * 2.0 ** k, np.inf) for k in range(-20, 10)]
    amaxes += [57344.0, 57344.5, 1.0, 0.875 * 512]
    for a in amaxes:
        k = orc.ds_tile_exponent(a)
        assert a <= 448.0 * 2.0 ** k
        assert a > 448.0 * 2.0 ** (k - 1)
    assert orc.ds_tile_exponent(0.0) == 0
    # the pages' bound: |x| <= 57344 gives a power-of-two scale <= 2^7
    assert orc.ds_tile_exponent(57344.0) == 7
    assert orc.ds_tile_exponent(1e-45) == -126   # clamped at the fp32 normal range
