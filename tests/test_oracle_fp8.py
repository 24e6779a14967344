"""Pins of the oracle's FP8 E4M3 keys (k8v4 format) against the format itself and
an independent implementation (PyTorch's float8_e4m3fn conversion)."""
import math

import numpy as np
import pytest

from oracle import fp8


def test_every_finite_code_round_trips():
    for b in range(256):
        if b in (0x7F, 0xFF):
            assert math.isnan(fp8.decode_byte(b))
            continue
        v = fp8.decode_byte(b)
        assert fp8.encode_value(v) == b, hex(b)


def test_values_of_the_format():
    assert fp8.decode_byte(0x38) == 1.0 and fp8.decode_byte(0xB8) == -1.0
    assert fp8.decode_byte(0x40) == 2.0
    assert fp8.decode_byte(0x7E) == 448.0 and fp8.decode_byte(0xFE) == -448.0
    assert fp8.decode_byte(0x08) == 2.0 ** -6  # smallest normal
    assert fp8.decode_byte(0x01) == 2.0 ** -9  # smallest subnormal
    assert fp8.decode_byte(0x07) == 7 * 2.0 ** -9
    assert fp8.decode_byte(0x00) == 0.0 and math.copysign(1.0, fp8.decode_byte(0x80)) < 0
    finite = sorted(fp8.decode_byte(b) for b in range(128) if b != 0x7F)
    assert len(set(finite)) == 127 and all(a < b for a, b in zip(finite, finite[1:]))


def test_ties_go_to_even_and_others_to_nearest():
    grid = [fp8.decode_byte(b) for b in range(0x7F)]  # 0 .. 448, increasing
    for b in range(len(grid) - 1):
        lo, hi = grid[b], grid[b + 1]
        mid = 0.5 * (lo + hi)
        expect = b if b % 2 == 0 else b + 1
        assert fp8.encode_value(mid) == expect
        assert fp8.encode_value(-mid) == 0x80 | expect
        assert fp8.encode_value(lo + 0.25 * (hi - lo)) == b
        assert fp8.encode_value(lo + 0.75 * (hi - lo)) == b + 1


def test_saturation_and_nan():
    for v in (448.0, 460.0, 464.0, 470.0, 480.0, 1e6, math.inf):
        assert fp8.encode_value(v) == 0x7E
        assert fp8.encode_value(-v) == 0xFE
    assert fp8.encode_value(math.nan) == 0x7F
    assert fp8.encode_value(2.0 ** -11) == 0x00  # below half the smallest subnormal
    assert fp8.encode_value(3 * 2.0 ** -11) == 0x01


def test_agrees_with_torch_float8_e4m3fn():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("no float8_e4m3fn in this torch")
    g = np.random.default_rng(8)
    x = np.concatenate([g.standard_normal(4000) * s for s in (0.01, 1.0, 30.0)])
    x = x[np.abs(x) < 448.0].astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(fp8.encode(x), ref)
    assert np.array_equal(fp8.decode(ref), torch.from_numpy(ref).view(torch.float8_e4m3fn).float().numpy())
