"""CPU oracle for the single-GPU MoE expert-layer hot path.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, fp64 restatement of
what the layer computes, written from the sglang PR reports that describe it:

* "Support DeepGEMM for standard MoE dispatch" (sglang PR #33128 report):
  compact / masked per-expert layouts, the static compact row bound, the
  ``-1`` padding rule for ``m_indices``, direct UE8M0 activation quantisation.
* "Add BF16 support to EP-MoE for DeepGEMM" (sglang PR #17392 report):
  the BF16 grouped-GEMM sequence GEMM(w13) -> SiLU(gate)*up -> GEMM(w2).
* "[Feature] Support BF16 and batch-invariant inference with DeepEP v2"
  (sglang PR #38160 report): ``expert_start`` / local-expert ranges, combine
  through stored slot pointers, bitwise batch invariance.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it.  It shares no code with the CUDA path and never
imports the product package; the product path never imports it.

Pinning status (what each function is checked against in ``tests/``):

* ``formats``: bf16 / e4m3 rounding against torch's own dtype casts over
  exhaustive bf16 sweeps; UE8M0 exponent against a brute-force search;
  1x32 (MXFP8) groups against torch's e4m3 cast with a brute-force minimal
  exponent, against the 1x128 routine on tiled blocks, and equal to 1x128
  where the four blocks of a group share their exponent; E2M1 (FP4) values
  against the E4M3 grid (pinned above): exactly the E4M3 values of at most
  two significant bits between 0.5 and 6, plus zero.
* ``layout``: the static compact bound against brute force over every
  routing of tiny problems; plan invariants (bijection, stability, ``-1``
  padding) on random routings.
* ``router``: selection against a keyed sort and brute force over tiny rows
  with ties; softmax against scipy's and torch's; logits against torch
  float64.
* ``requant``: an element-by-element restatement with torch's casts and a
  brute-force exponent search; exact round trip for power-of-two scales.
* ``moe``: layout-based forward == per-token loop (bitwise); k=1 single expert
  == a textbook SwiGLU MLP in torch float64; hand-computed small-integer
  weights; masked == compact (bitwise); MXFP8 weight dequantisation element
  by element with plain loops.
"""

from .formats import (  # noqa: F401
    BF16_MAX,
    E4M3_MAX,
    bf16_round,
    bf16_bits,
    e4m3_round,
    e4m3_bits,
    e4m3_from_bits,
    ue8m0_exponent,
    quant_fp8_1x128,
    dequant_1x128,
    quant_fp8_groups,
    dequant_groups,
    quant_mxfp8_1x32,
    e2m1_from_codes,
    unpack_fp4,
)
from .layout import (  # noqa: F401
    compact_all_tokens,
    use_masked_layout,
    plan_layout,
)
from .moe import (  # noqa: F401
    combine,
    dequant_fp8_weights,
    dequant_mx_weights,
    dequant_mxfp4_weights,
    expert_ffn,
    gemm1_act,
    gemm2,
    store_act,
    forward_layout,
    forward_per_token,
    silu,
)
from .requant import requant_block_ue8m0  # noqa: F401
from . import router  # noqa: F401
