"""Pins for the oracle's number formats (bf16 rounding, OCP E4M3 encoding, FP8 rows).

Each check compares the oracle with something other than itself: torch's CPU
conversions (library routines), a brute-force nearest-value search over all 256
E4M3 codes, and values fixed by the format definitions.
"""
import math
import struct

import numpy as np
import pytest
import torch

import oracle


def _f32(bits):
    return struct.unpack("<f", struct.pack("<I", bits & 0xFFFFFFFF))[0]


def _bits(f):
    return struct.unpack("<I", struct.pack("<f", f))[0]


# ----------------------------------------------------------------------------- bf16

def test_bf16_matches_torch_on_random_and_edge_values():
    rng = np.random.Generator(np.random.PCG64(11))
    bits = rng.integers(0, 2**32, size=200_000, dtype=np.uint64).astype(np.uint32)
    # ties, near-ties and carries into the exponent
    extra = []
    for base in (0x3F800000, 0x3F810000, 0x7F7F0000, 0x00010000, 0x80800000, 0x477F0000):
        for low in (0x7FFF, 0x8000, 0x8001, 0xFFFF, 0x0000, 0x0001):
            extra.append(base | low)
    bits = np.concatenate([bits, np.array(extra, np.uint32)])
    vals = bits.view(np.float32)
    finite = np.isfinite(vals)
    vals = vals[finite]
    ref = torch.from_numpy(vals.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ours = np.array([oracle.f32_to_bf16(float(v)) for v in vals[:40000]] +
                    [oracle.f32_to_bf16(float(v)) for v in vals[-len(extra):]], np.uint16)
    expect = np.concatenate([ref[:40000], ref[-len(extra):]])
    assert np.array_equal(ours, expect)


def test_bf16_special_values():
    assert oracle.f32_to_bf16(float("inf")) == 0x7F80
    assert oracle.f32_to_bf16(float("-inf")) == 0xFF80
    nan = oracle.f32_to_bf16(float("nan"))
    assert (nan & 0x7F80) == 0x7F80 and (nan & 0x007F) != 0
    # the largest finite float rounds up to infinity
    assert oracle.f32_to_bf16(_f32(0x7F7FFFFF)) == 0x7F80
    # exact ties go to the even upper half
    assert oracle.f32_to_bf16(_f32(0x3F808000)) == 0x3F80
    assert oracle.f32_to_bf16(_f32(0x3F818000)) == 0x3F82
    assert oracle.f32_to_bf16(-0.0) == 0x8000
    for b in (0x0000, 0x3F80, 0xBF80, 0x0001, 0x7F7F):
        assert _bits(oracle.bf16_to_f32(b)) == b << 16


# ----------------------------------------------------------------------------- e4m3

def _all_codes():
    """Values of every finite E4M3 code from the format definition, by brute force."""
    vals = {}
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            continue
        v = (m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
        vals[c] = -v if s else v
    return vals


CODES = _all_codes()


def _nearest_even(v):
    """Round v to the nearest finite E4M3 value; ties to the code with even mantissa; saturate."""
    if v > 448.0:
        return 0x7E
    if v < -448.0:
        return 0xFE
    best = None
    for c, cv in CODES.items():
        if (cv == 0.0) and (math.copysign(1.0, cv) != math.copysign(1.0, v)):
            continue  # keep the sign of zero
        d = abs(cv - v)
        if best is None or d < best[0] or (d == best[0] and (c & 1) == 0 and (best[1] & 1) == 1):
            best = (d, c)
    return best[1]


def test_e4m3_decode_matches_definition_and_torch():
    for c in range(256):
        ours = oracle.e4m3_to_f32(c)
        t = torch.tensor([c], dtype=torch.uint8).view(torch.float8_e4m3fn).float().item()
        if c in CODES:
            assert ours == CODES[c]
            assert ours == t
        else:
            assert math.isnan(ours) and math.isnan(t)


def test_e4m3_encode_brute_force_on_midpoints_and_neighbours():
    pts = set()
    finite = sorted(set(CODES.values()))
    for a, b in zip(finite[:-1], finite[1:]):
        mid = np.float32((a + b) / 2)  # E4M3 midpoints are exact in binary32
        pts.add(float(mid))
        pts.add(float(np.nextafter(mid, np.float32(np.inf))))
        pts.add(float(np.nextafter(mid, np.float32(-np.inf))))
        pts.add(float(np.float32(a)))
    pts.update([448.0, 449.0, 463.99, 464.0, 465.0, 1e30, -1e30, 2.0**-9, 2.0**-10, 3 * 2.0**-10,
                2.0**-11, 0.0, -0.0, 2.0**-6, 2.0**-6 - 2.0**-10])
    for v in pts:
        assert oracle.f32_to_e4m3(v) == _nearest_even(v), v


def test_e4m3_encode_matches_torch_on_random_in_range_values():
    rng = np.random.Generator(np.random.PCG64(5))
    mags = np.exp(rng.uniform(np.log(2.0**-12), np.log(448.0), size=30000)).astype(np.float32)
    vals = mags * rng.choice(np.array([-1, 1], np.float32), size=mags.size)
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = np.array([oracle.f32_to_e4m3(float(v)) for v in vals], np.uint8)
    assert np.array_equal(ours, ref)


def test_e4m3_saturates_and_keeps_nan():
    assert oracle.f32_to_e4m3(float("inf")) == 0x7E
    assert oracle.f32_to_e4m3(float("-inf")) == 0xFE
    assert oracle.f32_to_e4m3(float("nan")) & 0x7F == 0x7F


# ----------------------------------------------------------------------------- FP8 rows

def _torch_quantize(x_bits):
    """The 1x128 quantisation restated with torch CPU ops (fp32 division, library fp8 cast)."""
    x = torch.from_numpy(x_bits.view(np.int16).copy()).view(torch.bfloat16).float().view(-1, 128)
    amax = x.abs().amax(dim=1, keepdim=True)
    scale = amax / torch.tensor(448.0)
    q = (x / scale).to(torch.float8_e4m3fn).view(torch.uint8)
    return q.reshape(-1).numpy(), scale.reshape(-1).numpy()


def test_fp8_row_matches_torch_restatement():
    rng = np.random.Generator(np.random.PCG64(7))
    for H, sigma in ((1024, 1.0), (7168, 1.0), (256, 1e-3), (512, 300.0)):
        x = torch.from_numpy((rng.standard_normal(H) * sigma).astype(np.float32)).to(torch.bfloat16)
        bits = x.view(torch.int16).numpy().view(np.uint16)
        q, s = oracle.quantize_row_e4m3(bits)
        tq, ts = _torch_quantize(bits)
        assert np.array_equal(s.view(np.uint32), ts.view(np.uint32))
        assert np.array_equal(q, tq)


def test_fp8_row_block_max_hits_448_and_error_bound():
    rng = np.random.Generator(np.random.PCG64(8))
    x = torch.from_numpy(rng.standard_normal(7168).astype(np.float32)).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    q, s = oracle.quantize_row_e4m3(bits)
    xf = x.float().numpy().reshape(-1, 128)
    qv = np.array([oracle.e4m3_to_f32(int(c)) for c in q], np.float64).reshape(-1, 128)
    for b in range(xf.shape[0]):
        i = int(np.argmax(np.abs(xf[b])))
        assert q.reshape(-1, 128)[b, i] in (0x7E, 0xFE)
        # |q*scale - x| <= half an e4m3 step at q's binade, times the scale (+ fp32 slack)
        step = np.where(np.abs(qv[b]) >= 2.0**-6, 2.0 ** (np.floor(np.log2(np.maximum(np.abs(qv[b]), 2.0**-6))) - 3), 2.0**-9)
        err = np.abs(qv[b] * s[b] - xf[b])
        assert np.all(err <= (0.5 * step + 1e-6 * np.abs(qv[b])) * s[b] * (1 + 1e-6) + 1e-30)


def test_fp8_zero_block_and_signed_zero():
    bits = np.zeros(256, np.uint16)
    bits[3] = 0x8000  # -0 in the all-zero first block
    bits[128] = 0x3F80  # second block has amax 1
    bits[129] = 0x8000  # -0 in a block with a positive scale
    q, s = oracle.quantize_row_e4m3(bits)
    assert s[0] == 0.0 and q[0] == 0x00 and q[3] == 0x80
    assert s[1] == np.float32(1.0) / np.float32(448.0)
    assert q[128] == 0x7E and q[129] == 0x80 and q[130] == 0x00
