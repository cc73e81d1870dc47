"""Seeded synthetic inputs for the MoE expert layer.

This module only draws random inputs in the layer's storage formats; it holds
none of the layer's arithmetic.  Both the CUDA path and the CPU oracle consume
the exact bytes it returns.

* Activations x: bf16 ~ N(0, 1).
* Router: logits z [T, E_global] ~ N(0, 1) (plus log p_{pi(i)} with
  p_r ~ r^-s for the skewed "Zipf" popularity, pi a seeded permutation so
  popular experts are scattered); the top-k experts by logit (ties to the
  lower id), weights = softmax over the selected logits, stored fp32.  The
  router itself is not part of the layer; its output is the layer's input.
* FP8 weights: drawn directly in stored form.  Each 128x128 block gets a
  UE8M0 exponent s in {-12, -11} (byte s + 127), and its values are
  N(0, 0.02) * 2^-s clamped to +-448 and cast to E4M3 by torch's dtype cast.
  That matches FP8 quantisation of N(0, 0.02) weights at these scales without
  running the layer's quantisation rule here.
* BF16 weights: N(0, 0.02) cast to bf16.

Weights are seeded per expert (seed, expert), so any subset of experts is
reproducible on its own (the masked decode workload reuses the first experts
of the large-prefill weights).  Large weights are drawn on the GPU in chunks.
"""

import numpy as np
import torch

FP8_WEIGHT_EXPONENTS = (-12, -11)


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def activations(T, K, seed, device="cpu"):
    """x [T, K] bf16 ~ N(0, 1)."""
    g = _gen(seed, device)
    return torch.randn((T, K), generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def router_logits(T, E, seed, zipf_s=None):
    """Router logits [T, E] fp64 (numpy)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    z = rng.standard_normal((T, E))
    if zipf_s is not None:
        p = np.arange(1, E + 1, dtype=np.float64) ** (-zipf_s)
        p /= p.sum()
        perm = rng.permutation(E)
        z = z + np.log(p[perm])[None, :]
    return z


def topk_from_logits(z, topk):
    """Top-k expert ids (descending logit, ties to the lower id) and the
    softmax over the selected logits, as (int32 [T, k], fp32 [T, k])."""
    order = np.argsort(-z, axis=1, kind="stable")[:, :topk]
    sel = np.take_along_axis(z, order, axis=1)
    w = np.exp(sel - sel[:, :1])
    w = w / w.sum(axis=1, keepdims=True)
    return order.astype(np.int32), w.astype(np.float32)


def routing(T, E, topk, seed, zipf_s=None):
    """(topk_ids int32 [T, k], topk_weights fp32 [T, k]) as torch CPU tensors."""
    ids, w = topk_from_logits(router_logits(T, E, seed, zipf_s), topk)
    return torch.from_numpy(ids), torch.from_numpy(w)


def fp8_expert_weights(E, N, C, seed, device="cpu", first_expert=0):
    """FP8 weights for experts first_expert .. first_expert+E-1.

    Returns (w uint8 [E, N, C] E4M3 bytes, w_sf uint8 [E, N/128, C/128]
    UE8M0 bytes).
    """
    assert N % 128 == 0 and C % 128 == 0
    w = torch.empty((E, N, C), dtype=torch.uint8, device=device)
    sf = torch.empty((E, N // 128, C // 128), dtype=torch.uint8, device=device)
    rows_per_chunk = max(128, (1 << 26) // C // 128 * 128)
    for i in range(E):
        g = _gen(seed * 1_000_003 + first_expert + i, device)
        choice = torch.randint(0, len(FP8_WEIGHT_EXPONENTS), (N // 128, C // 128), generator=g, device=device)
        exps = torch.tensor(FP8_WEIGHT_EXPONENTS, device=device)[choice]
        sf[i] = (exps + 127).to(torch.uint8)
        for r0 in range(0, N, rows_per_chunk):
            r1 = min(N, r0 + rows_per_chunk)
            v = torch.randn((r1 - r0, C), generator=g, device=device, dtype=torch.float32) * 0.02
            mult = torch.exp2(-exps[r0 // 128:r1 // 128].to(torch.float32))
            v = v.view(-1, 128, C // 128, 128) * mult.view(-1, 1, C // 128, 1)
            v = v.clamp_(-448.0, 448.0).view(r1 - r0, C)
            w[i, r0:r1] = v.to(torch.float8_e4m3fn).view(torch.uint8)
    return w, sf


def mxfp8_expert_weights(E, N, C, seed, device="cpu", first_expert=0):
    """MXFP8 weights for experts first_expert .. first_expert+E-1: one UE8M0
    exponent per row and 32-column block.

    Returns (w uint8 [E, N, C] E4M3 bytes, w_sf uint8 [E, N, C/32] UE8M0
    bytes, row-major: the natural MX layout).
    """
    assert N % 128 == 0 and C % 128 == 0
    w = torch.empty((E, N, C), dtype=torch.uint8, device=device)
    sf = torch.empty((E, N, C // 32), dtype=torch.uint8, device=device)
    rows_per_chunk = max(128, (1 << 26) // C // 128 * 128)
    for i in range(E):
        g = _gen(seed * 1_000_003 + first_expert + i + 7919, device)
        choice = torch.randint(0, len(FP8_WEIGHT_EXPONENTS), (N, C // 32), generator=g, device=device)
        exps = torch.tensor(FP8_WEIGHT_EXPONENTS, device=device)[choice]
        sf[i] = (exps + 127).to(torch.uint8)
        for r0 in range(0, N, rows_per_chunk):
            r1 = min(N, r0 + rows_per_chunk)
            v = torch.randn((r1 - r0, C), generator=g, device=device, dtype=torch.float32) * 0.02
            mult = torch.exp2(-exps[r0:r1].to(torch.float32))
            v = (v.view(r1 - r0, C // 32, 32) * mult.view(r1 - r0, C // 32, 1)).clamp_(-448.0, 448.0)
            w[i, r0:r1] = v.view(r1 - r0, C).to(torch.float8_e4m3fn).view(torch.uint8)
    return w, sf


# FP4 E2M1 magnitude codes 0..7 (0, 0.5, 1, 1.5, 2, 3, 4, 6) drawn with these
# weights: a bell-shaped spread of codes, 6 kept rare.
FP4_CODE_WEIGHTS = (0.10, 0.20, 0.20, 0.15, 0.13, 0.10, 0.08, 0.04)
FP4_WEIGHT_EXPONENTS = (-9, -8)


def mxfp4_expert_weights(E, N, C, seed, device="cpu", first_expert=0):
    """MXFP4 weights for experts first_expert .. first_expert+E-1, drawn as
    codes: E2M1 codes packed two per byte (element 2j in the low nibble of
    byte j) and one UE8M0 exponent per row and 32-column block.

    Returns (w uint8 [E, N, C/2], w_sf uint8 [E, N, C/32], natural layout).
    """
    assert N % 128 == 0 and C % 128 == 0
    w = torch.empty((E, N, C // 2), dtype=torch.uint8, device=device)
    sf = torch.empty((E, N, C // 32), dtype=torch.uint8, device=device)
    probs = torch.tensor(FP4_CODE_WEIGHTS, dtype=torch.float32, device=device)
    rows_per_chunk = max(128, (1 << 26) // C // 128 * 128)
    for i in range(E):
        g = _gen(seed * 1_000_003 + first_expert + i + 104729, device)
        choice = torch.randint(0, len(FP4_WEIGHT_EXPONENTS), (N, C // 32), generator=g, device=device)
        sf[i] = (torch.tensor(FP4_WEIGHT_EXPONENTS, device=device)[choice] + 127).to(torch.uint8)
        for r0 in range(0, N, rows_per_chunk):
            r1 = min(N, r0 + rows_per_chunk)
            n = (r1 - r0) * C
            mag = torch.multinomial(probs, n, replacement=True, generator=g).view(r1 - r0, C)
            sign = torch.randint(0, 2, (r1 - r0, C), generator=g, device=device) * 8
            code = (mag + sign).to(torch.uint8)
            w[i, r0:r1] = code[:, 0::2] | (code[:, 1::2] << 4)
    return w, sf


def bf16_expert_weights(E, N, C, seed, device="cpu", first_expert=0):
    """BF16 weights [E, N, C] ~ N(0, 0.02)."""
    w = torch.empty((E, N, C), dtype=torch.bfloat16, device=device)
    rows_per_chunk = max(1, (1 << 26) // C)
    for i in range(E):
        g = _gen(seed * 1_000_003 + first_expert + i, device)
        for r0 in range(0, N, rows_per_chunk):
            r1 = min(N, r0 + rows_per_chunk)
            w[i, r0:r1] = (torch.randn((r1 - r0, C), generator=g, device=device, dtype=torch.float32) * 0.02).to(torch.bfloat16)
    return w


def probe_tokens(n_probe, K, E, topk, seed, zipf_s=None):
    """Fixed probe tokens for the batch-invariance sweep: x [n, K] bf16 and
    routing drawn from seeds that depend only on the probe index."""
    xs, ids, ws = [], [], []
    for p in range(n_probe):
        xs.append(activations(1, K, seed * 7919 + p))
        i, w = routing(1, E, topk, seed * 7919 + p, zipf_s)
        ids.append(i)
        ws.append(w)
    return torch.cat(xs), torch.cat(ids), torch.cat(ws)


# Workload recipes.  Sizes follow the published shapes of the pages'
# workloads; "seed" is fixed per workload.
WORKLOADS = {
    "tiny_fp8": dict(T=128, K=256, I=256, E_global=8, E_local=8, expert_start=0, topk=2,
                     dtype="fp8", layout="compact", zipf_s=None, seed=0x4D6F45_0001),
    "bf16_prefill": dict(T=4096, K=2048, I=768, E_global=128, E_local=128, expert_start=0, topk=8,
                         dtype="bf16", layout="compact", zipf_s=None, seed=0x4D6F45_0002),
    "fp8_prefill_zipf": dict(T=8192, K=7168, I=2048, E_global=256, E_local=256, expert_start=0, topk=8,
                             dtype="fp8", layout="compact", zipf_s=1.2, seed=0x4D6F45_0003),
    # profiling-sized FP8 prefill (1.4 GB of weights): same per-tile shape as
    # the large prefill, small enough for a full ncu capture
    "fp8_prefill_e32": dict(T=2048, K=7168, I=2048, E_global=32, E_local=32, expert_start=0, topk=8,
                            dtype="fp8", layout="compact", zipf_s=None, seed=0x4D6F45_0004),
    "fp8_masked_decode": dict(T=64, K=7168, I=2048, E_global=256, E_local=32, expert_start=0, topk=8,
                              dtype="fp8", layout="masked", zipf_s=None, seed=0x4D6F45_0003),
    # the MXFP8 variant (1x32 UE8M0 scales everywhere) of the two shapes above
    "mxfp8_prefill_zipf": dict(T=8192, K=7168, I=2048, E_global=256, E_local=256, expert_start=0, topk=8,
                               dtype="mxfp8", layout="compact", zipf_s=1.2, seed=0x4D6F45_0003),
    "mxfp8_masked_decode": dict(T=64, K=7168, I=2048, E_global=256, E_local=32, expert_start=0, topk=8,
                                dtype="mxfp8", layout="masked", zipf_s=None, seed=0x4D6F45_0003),
    # FP4 (E2M1) weights with 1x32 UE8M0 scales, MXFP8 activations
    "mxfp4_prefill_zipf": dict(T=8192, K=7168, I=2048, E_global=256, E_local=256, expert_start=0, topk=8,
                               dtype="mxfp4", layout="compact", zipf_s=1.2, seed=0x4D6F45_0003),
    "mxfp4_masked_decode": dict(T=64, K=7168, I=2048, E_global=256, E_local=32, expert_start=0, topk=8,
                                dtype="mxfp4", layout="masked", zipf_s=None, seed=0x4D6F45_0003),
}
