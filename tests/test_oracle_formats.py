"""Pins for oracle.formats against independent references.

* bf16 / E4M3 rounding: torch's own dtype casts (library routines), swept over
  every bf16 bit pattern.
* UE8M0 exponent: a brute-force search for the smallest admissible exponent.
* 1x128 quantisation: the bounds and invariants the direct-UE8M0 rule of
  "Support DeepGEMM for standard MoE dispatch" ("实现拆解" step 3) implies.
"""

import math

import numpy as np
import pytest
import torch

from oracle import formats as F


def all_bf16_values():
    bits = np.arange(1 << 16, dtype=np.uint32) << 16
    f = bits.view(np.float32)
    return f[np.isfinite(f)].astype(np.float64)


def test_bf16_round_matches_torch_cast_on_fp32():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 1 << 32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    # force exact ties and near-ties on a slice of the sample
    bits[: 1 << 16] = (np.arange(1 << 16, dtype=np.uint32) << 16) | 0x8000
    bits[1 << 16: 2 << 16] = (np.arange(1 << 16, dtype=np.uint32) << 16) | 0x7FFF
    f = bits.view(np.float32)
    f = f[np.isfinite(f) & (np.abs(f) <= np.float32(F.BF16_MAX))]
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ours = F.bf16_bits(F.bf16_round(f.astype(np.float64)))
    assert np.array_equal(ours, ref)


def test_bf16_round_direct_from_fp64_ties():
    # 1 + 2^-8 is exactly half-way between 1 and 1 + 2^-7 -> even (1.0);
    # adding 2^-40 breaks the tie upward, which rounding via fp32 would lose.
    assert F.bf16_round(1.0 + 2.0 ** -8) == 1.0
    assert F.bf16_round(1.0 + 2.0 ** -8 + 2.0 ** -40) == 1.0 + 2.0 ** -7
    assert F.bf16_round(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6
    assert F.bf16_round(-0.0) == 0.0 and math.copysign(1, F.bf16_round(-0.0)) < 0
    assert np.isinf(F.bf16_round(3.5e38))


@pytest.mark.parametrize("shift", [-12, -8, -3, 0, 3, 7, 9, 15])
def test_e4m3_round_and_bits_match_torch_cast(shift):
    v = all_bf16_values() * 2.0 ** shift
    v = v[np.abs(v) <= 464.0]                    # torch does not saturate above
    f = v.astype(np.float32)
    keep = f.astype(np.float64) == v             # exactly representable inputs only
    f, v = f[keep], v[keep]
    ref = torch.from_numpy(f.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    q = F.e4m3_round(v)
    assert np.all(np.abs(q) <= F.E4M3_MAX)
    assert np.array_equal(F.e4m3_bits(q), ref)
    assert np.array_equal(F.e4m3_from_bits(ref), q)


def test_e4m3_saturates_and_grid_constants():
    assert F.e4m3_round(465.0) == 448.0 and F.e4m3_round(-1e6) == -448.0
    assert F.e4m3_round(2.0 ** -10) == 0.0                  # tie between 0 and 2^-9 -> 0
    assert F.e4m3_round(1.5 * 2.0 ** -9) == 2.0 ** -8        # tie 1 / 2 steps -> 2 steps
    assert F.e4m3_from_bits(0x7E) == 448.0 and F.e4m3_from_bits(0x01) == 2.0 ** -9
    assert F.e4m3_from_bits(0x08) == 2.0 ** -6 and np.isnan(F.e4m3_from_bits(0x7F))
    codes = np.arange(256, dtype=np.uint8)
    vals = F.e4m3_from_bits(codes)
    ok = ~np.isnan(vals)
    assert np.array_equal(F.e4m3_bits(vals[ok]), codes[ok])


def brute_force_exponent(amax):
    if amax == 0:
        return -127
    s = -200
    while amax > 448.0 * 2.0 ** s:
        s += 1
    return max(-127, min(127, s))


def test_ue8m0_exponent_is_minimal_over_all_bf16():
    v = all_bf16_values()
    v = np.unique(np.abs(v))
    ours = F.ue8m0_exponent(v)
    ref = np.array([brute_force_exponent(a) for a in v])
    assert np.array_equal(ours, ref)


def test_quant_fp8_1x128_invariants():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((64, 512)) * np.exp2(rng.integers(-20, 20, size=(64, 1)))
    x[3, 128:256] = 0.0                              # an all-zero group
    x[5, :128] = 448.0 * 2.0 ** 3                    # amax exactly on a power boundary
    x = F.bf16_round(x)
    q, s = F.quant_fp8_1x128(x)
    assert np.all(np.abs(q) <= 448.0)
    amax = np.abs(x.reshape(64, 4, 128)).max(axis=2)
    assert np.all(amax <= 448.0 * np.exp2(s))
    lower = amax > 448.0 * np.exp2(s - 1)
    assert np.all(lower | (s == -127))
    assert s[3, 1] == -127 and s[5, 0] == 3
    # the largest element of each non-zero group lands in the top binade
    top = np.abs(q.reshape(64, 4, 128)).max(axis=2)
    assert np.all((top >= 224.0) | (amax == 0))
    # values already on the grid are reproduced exactly (idempotence of the
    # dequantised values; the exponent may drop by one when the group max
    # rounded down to exactly 224 * 2^s)
    deq = F.dequant_1x128(q, s)
    q2, s2 = F.quant_fp8_1x128(deq)
    assert np.array_equal(F.dequant_1x128(q2, s2), deq)
    assert np.all((s2 == s) | (s2 == s - 1))
    # relative error bounded by half an E4M3 step (2^-4) of the scale-normalised value
    err = np.abs(deq - x).reshape(64, 4, 128)
    bound = np.maximum(np.abs(x).reshape(64, 4, 128) * 2.0 ** -4, 2.0 ** -10 * np.exp2(s)[..., None])
    assert np.all(err <= bound)


def test_quant_groups_are_independent():
    rng = np.random.default_rng(8)
    x = F.bf16_round(rng.standard_normal((4, 384)))
    q, s = F.quant_fp8_1x128(x)
    x2 = x.copy()
    x2[:, 128:256] *= 1000.0
    q2, s2 = F.quant_fp8_1x128(x2)
    assert np.array_equal(q[:, :128], q2[:, :128]) and np.array_equal(q[:, 256:], q2[:, 256:])
    assert np.array_equal(s[:, [0, 2]], s2[:, [0, 2]])
