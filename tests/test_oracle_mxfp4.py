"""Pins for the MXFP4 (FP4 E2M1 weights, 1x32 UE8M0 scales) parts of the
oracle, against things other than the oracle's own decode:

* the E2M1 grid equals what its format parameters (two significant bits,
  normal exponents 0..2, subnormal step 1/2, no inf / NaN) select from the
  E4M3 grid, which test_oracle_formats pins against torch's own cast;
* the nibble order of the packing, byte by byte for all 256 bytes;
* dequantisation element by element with plain loops;
* the layer with MXFP4 weights: layout path == per-token loop (bitwise), and
  activations stored exactly as the MXFP8 path stores them.
"""

import math

import numpy as np

import oracle
import synth


def test_e2m1_grid_from_format_parameters():
    e4m3 = oracle.e4m3_from_bits(np.arange(256, dtype=np.uint8))
    mags = np.unique(np.abs(e4m3[np.isfinite(e4m3)]))
    normal = [v for v in mags if 1.0 <= v <= 6.0 and (2 * v / 2.0 ** math.floor(math.log2(v))) % 1 == 0]
    subnormal = [v for v in mags if v < 1.0 and (2 * v) % 1 == 0]
    expected = sorted(set(normal) | set(subnormal))
    got = oracle.e2m1_from_codes(np.arange(16))
    assert sorted(np.abs(got[:8]).tolist()) == expected == np.abs(got[:8]).tolist()   # codes 0..7 ascending
    assert np.array_equal(got[8:], -got[:8]) and np.signbit(got[8])                  # sign bit 3, -0 at 8
    assert len(expected) == 8 and max(expected) == 6.0


def test_unpack_fp4_nibble_order_all_bytes():
    codes = oracle.unpack_fp4(np.arange(256, dtype=np.uint8)[None, :])[0]
    for b in range(256):
        assert codes[2 * b] == b % 16 and codes[2 * b + 1] == b // 16


def test_dequant_mxfp4_weights_brute_force():
    rng = np.random.default_rng(8)
    E, N, C = 2, 128, 256
    wp = rng.integers(0, 256, size=(E, N, C // 2), dtype=np.uint8)
    we = rng.integers(-20, 20, size=(E, N, C // 32))
    got = oracle.dequant_mxfp4_weights(wp, we)
    mag = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for e in range(E):
        for n in range(0, N, 7):
            for c in range(0, C, 3):
                byte = int(wp[e, n, c // 2])
                code = byte & 15 if c % 2 == 0 else byte >> 4
                v = (-1.0 if code & 8 else 1.0) * mag[code & 7]
                assert got[e, n, c] == v * math.ldexp(1.0, int(we[e, n, c // 32])), (e, n, c)


def test_layer_with_mxfp4_weights_equals_per_token_loop():
    T, K, I, E_global, E_local, es, topk, seed = 40, 256, 256, 6, 4, 1, 3, 5
    x = synth.activations(T, K, seed).float().numpy().astype(np.float64)
    ids, w = synth.routing(T, E_global, topk, seed)
    ids = ids.numpy().copy()
    ids[::7, 0] = -1
    w13p, w13s = synth.mxfp4_expert_weights(E_local, 2 * I, K, seed)
    w2p, w2s = synth.mxfp4_expert_weights(E_local, K, I, seed + 1)
    w13 = oracle.dequant_mxfp4_weights(w13p.numpy(), w13s.numpy().astype(np.int64) - 127)
    w2 = oracle.dequant_mxfp4_weights(w2p.numpy(), w2s.numpy().astype(np.int64) - 127)
    ref = oracle.forward_per_token(x, w13, w2, ids, w.numpy(), "mxfp4", E_global, es)
    for layout in ("compact", "masked"):
        out = oracle.forward_layout(x, w13, w2, ids, w.numpy(), "mxfp4", E_global, es, layout=layout)
        assert np.array_equal(out, ref), layout
    assert np.count_nonzero(ref) > 0.9 * ref.size
    # activations and h are stored exactly as the MXFP8 path stores them
    a4, _ = oracle.store_act(x, "mxfp4")
    a8, _ = oracle.store_act(x, "mxfp8")
    assert np.array_equal(a4, a8)
