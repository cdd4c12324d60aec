"""The oracle's number formats against the OCP format definitions, PyTorch's own float8
cast and an exhaustive nearest-value search."""
import numpy as np
import pytest
import torch

import brute
from oracle import codecs



def test_e4m3_known_values():
    d = codecs.e4m3_decode(np.array([0x00, 0x01, 0x07, 0x08, 0x38, 0x7E, 0xFE, 0x80, 0xB8]))
    assert d.tolist() == [0.0, 2.0 ** -9, 7 * 2.0 ** -9, 2.0 ** -6, 1.0, 448.0, -448.0, -0.0,
                          -1.0]
    assert np.isnan(codecs.e4m3_decode(np.array([0x7F, 0xFF]))).all()


def test_e4m3_decode_matches_table_and_torch():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    ours = codecs.e4m3_decode(codes)
    table = np.array([brute.e4m3_value(int(c)) for c in codes])
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(ours, table)
    assert np.array_equal(ours, lib)


def test_e4m3_roundtrip_all_codes():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    assert np.array_equal(codecs.e4m3_encode(codecs.e4m3_decode(codes)), codes)


def test_e4m3_ties_and_saturation():
    pos = sorted({brute.e4m3_value(c) for c in range(0x7F)})
    mids = [(a + b) / 2 for a, b in zip(pos[:-1], pos[1:])]
    mids += [448.0, 460.0, 464.0, 470.0, 1e9, float(2.0 ** -10), 3 * 2.0 ** -11]
    v = np.array(mids + [-m for m in mids], dtype=np.float64)
    ours = codecs.e4m3_encode(v)
    ref = np.array([brute.e4m3_round(float(x)) for x in v], dtype=np.uint8)
    assert np.array_equal(ours, ref)


def test_e4m3_encode_matches_torch_cast_random():
    rng = np.random.default_rng(5)
    v = np.concatenate([
        rng.standard_normal(200000).astype(np.float32) * 100,
        rng.standard_normal(50000).astype(np.float32) * 2.0 ** -7,     # subnormal range
        rng.uniform(-448, 448, 50000).astype(np.float32),
    ])
    ours = codecs.e4m3_encode(v)
    lib = torch.from_numpy(np.clip(v, -448, 448)).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()
    assert np.array_equal(ours, lib)


def test_e2m1_table_and_unpack():
    vals = codecs.e2m1_decode(np.arange(16))
    assert vals[:8].tolist() == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert vals[8:].tolist() == [-0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]
    assert vals.tolist() == [brute.e2m1_value(c) for c in range(16)]
    packed = np.array([[0x21, 0xF7]], dtype=np.uint8)
    assert codecs.unpack_e2m1(packed).tolist() == [[1, 2, 7, 15]]
