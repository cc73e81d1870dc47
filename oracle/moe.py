"""The MoE expert layer, end to end, in fp64 (oracle; test use only).

Sequence (the BF16 run function printed in "Add BF16 support to EP-MoE for
DeepGEMM" (sglang PR #17392 report), section "关键源码片段" deep_gemm.py, and
the FP8 variant of "Support DeepGEMM for standard MoE dispatch" (sglang PR
#33128 report), "实现拆解" steps 1-3):

  1. layout      tokens -> per-expert rows (``layout.plan_layout``)
  2. quant       FP8: 1x128 UE8M0 quantisation of x; BF16: x as is
  3. GEMM1+act   g = a W1^T, u = a W3^T, h = silu(g) * u       (w13 = [W1; W3])
  4. GEMM2       y = h W2^T, stored as bf16
  5. combine     out[t] = sum_j w[t, j] * y[src2dst[t, j]], stored as bf16

Readings adopted where the reports are silent:

* w13[e] stacks the gate rows W1 (rows 0..I-1) above the up rows W3 (rows
  I..2I-1); the SiLU step of the printed run function splits the GEMM output
  in two halves of N/2 columns.
* g and u stay unrounded (fused activation); h is then stored in the GEMM2
  input format: FP8 with 1x128 UE8M0 scales (same rule as the activations)
  on the FP8 path, bf16 on the BF16 path.  y is stored as bf16 (the printed
  run function's down-projection output is bf16).
* The top-k weight is applied in the combine, after GEMM2 (fp32 weights).
* Weights are given per *local* expert: w13 [E_local, 2I, K], w2
  [E_local, K, I]; FP8 weights carry one UE8M0 exponent per 128x128 block.
* MXFP8 (dtype "mxfp8"): every scale covers 1x32 instead -- activations and
  h per row and 32-column block, weights per row and 32-column block along
  the reduction dimension -- with the same exponent rule.
* MXFP4 (dtype "mxfp4"): the weights are FP4 E2M1 with 1x32 UE8M0 scales;
  activations and h are MXFP8.

All sums are fp64.  ``forward_layout`` follows the layout path;
``forward_per_token`` computes the same layer one token at a time with no
layout at all, and the two must agree bitwise.
"""

import numpy as np

from .formats import (bf16_round, dequant_1x128, dequant_groups, e2m1_from_codes, e4m3_from_bits, quant_fp8_1x128,
                      quant_mxfp8_1x32, unpack_fp4)
from .layout import plan_layout, use_masked_layout


def silu(g):
    """silu(g) = g / (1 + exp(-g)) in fp64."""
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


def dequant_fp8_weights(w_bytes, w_exp):
    """FP8 weights [E, N, C] (E4M3 bytes) with 128x128 block exponents
    [E, N/128, C/128] -> fp64 values."""
    w = e4m3_from_bits(w_bytes)
    E, N, C = w.shape
    s = np.asarray(w_exp, dtype=np.int64)
    scale = np.ldexp(1.0, s)                                    # [E, N/128, C/128]
    return (w.reshape(E, N // 128, 128, C // 128, 128) * scale[:, :, None, :, None]).reshape(E, N, C)


def dequant_mx_weights(w_bytes, w_exp):
    """MXFP8 weights [E, N, C] (E4M3 bytes) with one exponent per row and
    32-column block, [E, N, C/32] -> fp64 values."""
    w = e4m3_from_bits(w_bytes)
    E, N, C = w.shape
    scale = np.ldexp(1.0, np.asarray(w_exp, dtype=np.int64))   # [E, N, C/32]
    return (w.reshape(E, N, C // 32, 32) * scale[..., None]).reshape(E, N, C)


def dequant_mxfp4_weights(w_packed, w_exp):
    """MXFP4 weights: E2M1 codes packed two per byte, [E, N, C/2] (element 2j
    in the low nibble of byte j), with one exponent per row and 32-column
    block, [E, N, C/32] -> fp64 values [E, N, C]."""
    w = e2m1_from_codes(unpack_fp4(w_packed))
    E, N, C = w.shape
    scale = np.ldexp(1.0, np.asarray(w_exp, dtype=np.int64))   # [E, N, C/32]
    return (w.reshape(E, N, C // 32, 32) * scale[..., None]).reshape(E, N, C)


def store_act(x, dtype):
    """Quantise activation rows to the GEMM input format; returns the fp64
    values the GEMM consumes and, for FP8 / MXFP8, the (q, s) pair."""
    if dtype == "fp8":
        q, s = quant_fp8_1x128(x)
        return dequant_1x128(q, s), (q, s)
    if dtype in ("mxfp8", "mxfp4"):          # MXFP4 weights keep MXFP8 activations
        q, s = quant_mxfp8_1x32(x)
        return dequant_groups(q, s, 32), (q, s)
    if dtype == "bf16":
        v = bf16_round(x)
        return v, (v, None)
    raise ValueError(dtype)


def gemm1_act(a, w13_e):
    """GEMM1 + activation on rows a [R, K] (fp64 values in the GEMM input
    format): returns (g, u, h) with h = silu(g) * u, all unrounded fp64."""
    I = w13_e.shape[0] // 2
    g = a @ w13_e[:I].T
    u = a @ w13_e[I:].T
    return g, u, silu(g) * u


def gemm2(h_in, w2_e):
    """GEMM2 on rows h_in [R, I] (stored h values): y = h W2^T rounded to bf16."""
    return bf16_round(h_in @ w2_e.T)


def combine(y, src2dst, topk_weights):
    """out[t] = bf16(sum_j w[t, j] * y[src2dst[t, j]]) over j with src2dst >= 0,
    summed in fp64 in j order; tokens with no destination get 0."""
    T, k = src2dst.shape
    out = np.zeros((T, y.shape[1]))
    for t in range(T):
        acc = np.zeros(y.shape[1])
        for j in range(k):
            d = src2dst[t, j]
            if d >= 0:
                acc = acc + float(topk_weights[t, j]) * y[d]
        out[t] = bf16_round(acc)
    return out


def expert_ffn(a, w13_e, w2_e, dtype, keep=False):
    """One expert on rows ``a`` [R, K] (already in the GEMM input format,
    fp64 values).  w13_e [2I, K], w2_e [K, I] fp64.  Returns y [R, K] (bf16
    values) and, with keep=True, a dict of the intermediates."""
    g, u, h = gemm1_act(a, w13_e)
    h_in, h_stored = store_act(h, dtype)
    y_acc = h_in @ w2_e.T
    y = bf16_round(y_acc)
    if keep:
        return y, {"g": g, "u": u, "h": h, "h_in": h_in, "h_stored": h_stored, "y_acc": y_acc}
    return y


def _check_shapes(x, w13, w2, topk_ids, topk_weights):
    T, K = x.shape
    E_l, N2, K2 = w13.shape
    if K2 != K or w2.shape != (E_l, K, N2 // 2):
        raise ValueError("weight shapes do not match x")
    if topk_ids.shape != topk_weights.shape or topk_ids.shape[0] != T:
        raise ValueError("routing shapes do not match x")
    return T, K, E_l, N2 // 2


def forward_layout(x, w13, w2, topk_ids, topk_weights, dtype, E_global, expert_start=0,
                   layout="auto", max_m=None, block_e=128, keep=False):
    """The whole layer through the per-expert layout.

    x [T, K] fp64 (bf16 values); w13 [E_local, 2I, K], w2 [E_local, K, I]
    fp64 (dequantised weights); topk_ids int [T, k]; topk_weights [T, k]
    (fp32 values).  dtype "fp8", "mxfp8", "mxfp4" or "bf16".  Returns out [T, K] (bf16 values)
    and, with keep=True, a dict with the plan and every stored intermediate.
    """
    x = np.asarray(x, dtype=np.float64)
    topk_ids = np.asarray(topk_ids)
    topk_weights = np.asarray(topk_weights, dtype=np.float64)
    T, K, E_l, I = _check_shapes(x, w13, w2, topk_ids, topk_weights)
    if layout == "auto":
        layout = "masked" if use_masked_layout(E_global, E_l) else "compact"
    if layout == "masked" and max_m is None:
        max_m = T
    plan = plan_layout(topk_ids, E_global, E_l, expert_start, layout, block_e, max_m)
    src2dst = plan["src2dst"]
    rows = plan["all_tokens"] if layout == "compact" else E_l * max_m

    # 2. quantise each token once, then scatter it to all its destination rows
    x_in, x_stored = store_act(x, dtype)
    a = np.full((rows, K), np.nan)          # rows without a token stay undefined
    for t in range(T):
        for j in range(topk_ids.shape[1]):
            d = src2dst[t, j]
            if d >= 0:
                a[d] = x_in[t]

    # 3-4. every expert on its own rows
    y = np.full((rows, K), np.nan)
    h_in = np.full((rows, I), np.nan)
    for e in range(E_l):
        if layout == "compact":
            r = np.flatnonzero(plan["m_indices"] == e)
        else:
            r = e * max_m + np.arange(plan["masked_m"][e])
        if r.size == 0:
            continue
        y_e, inter = expert_ffn(a[r], w13[e], w2[e], dtype, keep=True)
        y[r] = y_e
        h_in[r] = inter["h_in"]

    # 5. weighted combine in token order, fixed j order
    out = combine(y, src2dst, topk_weights)
    if keep:
        return out, {"plan": plan, "layout": layout, "x_in": x_in, "x_stored": x_stored,
                     "a": a, "h_in": h_in, "y": y, "max_m": max_m}
    return out


def forward_per_token(x, w13, w2, topk_ids, topk_weights, dtype, E_global, expert_start=0):
    """The same layer as sum_j w_j * expert_{e_j}(x_t), one token at a time,
    with no layout: the check that the layout bookkeeping adds nothing."""
    x = np.asarray(x, dtype=np.float64)
    topk_ids = np.asarray(topk_ids)
    topk_weights = np.asarray(topk_weights, dtype=np.float64)
    T, K, E_l, I = _check_shapes(x, w13, w2, topk_ids, topk_weights)
    out = np.zeros((T, K))
    for t in range(T):
        x_t, _ = store_act(x[t:t + 1], dtype)
        acc = np.zeros(K)
        for j in range(topk_ids.shape[1]):
            gid = int(topk_ids[t, j])
            e = gid - expert_start
            if gid < 0 or gid >= E_global or not 0 <= e < E_l:
                continue
            acc = acc + topk_weights[t, j] * expert_ffn(x_t, w13[e], w2[e], dtype)[0]
        out[t] = bf16_round(acc)
    return out
