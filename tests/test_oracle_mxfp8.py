"""Pins for the MXFP8 (1x32 UE8M0) parts of the oracle, against things other
than the oracle's own group routine:

* every 32-column block's exponent is the minimal one, found by brute force
  over exact powers of two, and the stored values are torch's own e4m3 cast
  of x * 2^-s (exact power-of-two scaling, nothing to saturate);
* a 32-column block quantised on its own equals the 1x128 routine (pinned in
  test_oracle_formats) applied to that block tiled four times;
* where the four 32-column blocks of a 128-column group share the group's
  exponent, MXFP8 and 1x128 give the same bytes;
* MXFP8 weight dequantisation element by element with plain loops.
"""

import math

import numpy as np
import torch

import oracle
from oracle import formats as F


def _groups_with_edge_values(R, C, seed):
    rng = np.random.default_rng(seed)
    x = F.bf16_round(rng.standard_normal((R, C)) * np.exp2(rng.integers(-20, 20, size=(R, C // 32)))
                     .repeat(32, axis=1))
    x[0, :32] = 0.0                                # all-zero block
    x[1, 32:64] = 1e-39                            # bf16 subnormals
    x[2, :32] = 448.0 * 8                          # amax exactly 448 * 2^3
    x[2, 32:64] = -448.0 * 8 * (1 + 2.0 ** -7)     # just above: one more exponent
    x[3, 64:96] = 3.0e38                           # near the bf16 maximum
    return x


def test_mx_exponent_is_brute_force_minimal_and_bytes_match_torch():
    x = _groups_with_edge_values(8, 256, 1)
    q, s = oracle.quant_mxfp8_1x32(x)
    assert s.shape == (8, 8)
    for r in range(8):
        for b in range(8):
            blk = x[r, 32 * b:32 * b + 32]
            amax = float(np.abs(blk).max())
            e = -127
            while e < 127 and amax > 448.0 * math.ldexp(1.0, e):
                e += 1
            assert s[r, b] == e, (r, b)
            ref = torch.from_numpy(blk * math.ldexp(1.0, -e)).to(torch.float8_e4m3fn).to(torch.float64).numpy()
            assert np.array_equal(q[r, 32 * b:32 * b + 32], ref), (r, b)
    assert s[2, 0] == 3 and s[2, 1] == 4 and s[0, 0] == -127


def test_mx_block_equals_1x128_of_the_block_tiled():
    x = _groups_with_edge_values(6, 384, 2)
    q, s = oracle.quant_mxfp8_1x32(x)
    for r in range(6):
        for b in range(384 // 32):
            blk = x[r, 32 * b:32 * b + 32]
            q4, s4 = oracle.quant_fp8_1x128(np.tile(blk, 4)[None, :])
            assert s4[0, 0] == s[r, b]
            assert np.array_equal(q4[0, :32], q[r, 32 * b:32 * b + 32])


def test_mx_equals_1x128_where_blocks_share_the_exponent():
    rng = np.random.default_rng(3)
    x = F.bf16_round(rng.uniform(-1.0, 1.0, size=(5, 512)))
    x[:, ::32] = 1.5                               # every 32-block holds the group amax
    q1, s1 = oracle.quant_fp8_1x128(x)
    q32, s32 = oracle.quant_mxfp8_1x32(x)
    assert np.array_equal(q1, q32)
    assert np.array_equal(np.repeat(s1, 4, axis=1), s32)
    # and the dequantised values agree
    assert np.array_equal(oracle.dequant_1x128(q1, s1), oracle.dequant_groups(q32, s32, 32))


def test_dequant_mx_weights_brute_force():
    rng = np.random.default_rng(6)
    E, N, C = 2, 128, 256
    wb = rng.integers(0, 256, size=(E, N, C), dtype=np.uint8)
    wb[(wb & 0x7F) == 0x7F] = 0x38                          # no NaN codes
    we = rng.integers(-20, 20, size=(E, N, C // 32))
    got = oracle.dequant_mx_weights(wb, we)
    for e in range(E):
        for n in range(0, N, 5):
            for c in range(0, C, 3):
                b = int(wb[e, n, c])
                sign = -1.0 if b & 0x80 else 1.0
                ef, mf = (b >> 3) & 0xF, b & 7
                v = sign * (mf / 8 * 2.0 ** -6 if ef == 0 else (1 + mf / 8) * 2.0 ** (ef - 7))
                assert got[e, n, c] == v * math.ldexp(1.0, int(we[e, n, c // 32])), (e, n, c)


def test_store_act_mxfp8_equals_fp8_store_of_tiled_blocks():
    """The layer's MXFP8 storage step (activations and h) per 32-column block
    equals the 1x128 storage step on that block tiled four times."""
    x = _groups_with_edge_values(4, 256, 4)
    vals, (q, s) = oracle.store_act(x, "mxfp8")
    assert s.shape == (4, 8)
    for r in range(4):
        for b in range(8):
            blk = x[r, 32 * b:32 * b + 32]
            v4, _ = oracle.store_act(np.tile(blk, 4)[None, :], "fp8")
            assert np.array_equal(vals[r, 32 * b:32 * b + 32], v4[0, :32])
