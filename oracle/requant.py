"""Load-time requantisation of block-scaled FP8 weights to UE8M0 scales
(oracle; test use only).

"Support DeepGEMM for standard MoE dispatch" (sglang PR #33128 report),
"实现拆解" step 1 and "关键源码片段" fp8.py: the standard MoE layer passes
both expert weight tensors (w13 and w2) with their 128x128 block scales to a
requantisation routine that produces UE8M0-scaled FP8 weights for the grouped
GEMMs, with bfloat16 as the intermediate ("output_dtype=torch.bfloat16").
The routine's body is not shown.  Reading adopted (the plainest one the call
supports, and the same power-of-two rule the layer uses for activations):

  1. dequantise each element: v = bf16( fp32(q) * s ), the product taken in
     fp32 (round to nearest even) and then rounded to bf16;
  2. per 128x128 block, the UE8M0 exponent e = smallest integer with
     amax(|v|) <= 448 * 2^e (clamped to [-127, 127], -127 for an all-zero
     block);
  3. requantise: q' = e4m3(v * 2^-e), round to nearest even, saturating.

Inputs are finite (no NaN codes).
"""

import numpy as np

from .formats import bf16_round, e4m3_bits, e4m3_from_bits, e4m3_round, ue8m0_exponent


def requant_block_ue8m0(w_bytes, scale):
    """w_bytes uint8 [E, N, C] E4M3 codes; scale float32 [E, N/128, C/128]
    (the dequantisation multiplier of each 128x128 block).  Returns (w_out
    uint8 [E, N, C], exp int64 [E, N/128, C/128]); the scale byte stored is
    exp + 127."""
    w = e4m3_from_bits(w_bytes)                       # exact fp64 values of the codes
    E, N, C = w.shape
    s = np.asarray(scale, dtype=np.float32)
    s_full = np.repeat(np.repeat(s, 128, axis=1), 128, axis=2)
    prod = (w.astype(np.float32) * s_full).astype(np.float64)     # fp32 product, RNE
    v = bf16_round(prod)
    blocks = np.abs(v).reshape(E, N // 128, 128, C // 128, 128).max(axis=(2, 4))
    e = ue8m0_exponent(blocks)
    e_full = np.repeat(np.repeat(e, 128, axis=1), 128, axis=2)
    q = e4m3_round(v * np.ldexp(1.0, -e_full))
    return e4m3_bits(q), e
