"""Pins for oracle.requant: an element-by-element restatement with torch's
own casts and a brute-force exponent search, and the exact round trip when
the input scales are already powers of two."""

import math

import numpy as np
import torch

import oracle
from oracle import requant as RQ


def _weights(seed, E=2, N=256, C=384):
    rng = np.random.default_rng(seed)
    w = rng.integers(0, 256, size=(E, N, C), dtype=np.uint8)
    w[(w & 0x7F) == 0x7F] = 0x3A                   # no NaN codes
    return w


def test_requant_matches_elementwise_restatement():
    w = _weights(1)
    rng = np.random.default_rng(2)
    s = (rng.uniform(1.0, 2.0, size=(2, 2, 3)) * np.exp2(rng.integers(-14, -9, size=(2, 2, 3)))).astype(np.float32)
    s[1, 1, 2] = 0.0                                 # an all-zero block
    out, e = RQ.requant_block_ue8m0(w, s)
    vals = torch.from_numpy(w.copy()).view(torch.float8_e4m3fn).float()
    for ex in range(2):
        for nb in range(2):
            for cb in range(3):
                blk = vals[ex, nb * 128:(nb + 1) * 128, cb * 128:(cb + 1) * 128]
                v = (blk * torch.tensor(float(s[ex, nb, cb]), dtype=torch.float32)).to(torch.bfloat16).double()
                amax = float(v.abs().max())
                k = -127
                while k < 127 and amax > 448.0 * 2.0 ** k:
                    k += 1
                assert e[ex, nb, cb] == k
                ref = (v * 2.0 ** -k).float().to(torch.float8_e4m3fn).view(torch.uint8).numpy()
                got = out[ex, nb * 128:(nb + 1) * 128, cb * 128:(cb + 1) * 128]
                assert np.array_equal(got, ref), (ex, nb, cb)


def test_power_of_two_scales_round_trip_exactly():
    w = _weights(3)
    rng = np.random.default_rng(4)
    s = np.exp2(rng.integers(-14, -9, size=(2, 2, 3))).astype(np.float32)
    out, e = RQ.requant_block_ue8m0(w, s)
    before = oracle.dequant_fp8_weights(w, np.log2(s).astype(np.int64))
    after = oracle.dequant_fp8_weights(out, e)
    assert np.array_equal(before, after)
    # the exponent never exceeds the input scale's (the block amax can only be
    # below 448 * s)
    assert np.all(e <= np.log2(s))
