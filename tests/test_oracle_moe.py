"""Pins for oracle.moe against things other than itself:

* the layout path equals a per-token loop sum_j w_j * expert_{e_j}(x) with no
  layout at all (bitwise), for FP8, MXFP8 and BF16, compact and masked;
* masked and compact layouts agree end to end (bitwise) -- the property the
  "Support DeepGEMM for standard MoE dispatch" report's end-to-end test checks;
* k = 1 through a single expert is a textbook SwiGLU MLP, checked against
  torch float64 (torch.nn.functional.silu and matmul);
* permutation weights give outputs that can be written down by hand, which
  catches a swapped gate/up, a transposed operand or a dropped combine term.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from oracle import formats as F
import synth


def small_problem(dtype, T=40, K=256, I=256, E_global=6, E_local=4, expert_start=1, topk=3, seed=5):
    x = synth.activations(T, K, seed).float().numpy().astype(np.float64)
    ids, w = synth.routing(T, E_global, topk, seed)
    ids = ids.numpy().copy()
    ids[::7, 0] = -1                                 # a few dropped assignments
    if dtype == "fp8":
        w13b, w13s = synth.fp8_expert_weights(E_local, 2 * I, K, seed)
        w2b, w2s = synth.fp8_expert_weights(E_local, K, I, seed + 1)
        w13 = oracle.dequant_fp8_weights(w13b.numpy(), w13s.numpy().astype(np.int64) - 127)
        w2 = oracle.dequant_fp8_weights(w2b.numpy(), w2s.numpy().astype(np.int64) - 127)
    elif dtype == "mxfp8":
        w13b, w13s = synth.mxfp8_expert_weights(E_local, 2 * I, K, seed)
        w2b, w2s = synth.mxfp8_expert_weights(E_local, K, I, seed + 1)
        w13 = oracle.dequant_mx_weights(w13b.numpy(), w13s.numpy().astype(np.int64) - 127)
        w2 = oracle.dequant_mx_weights(w2b.numpy(), w2s.numpy().astype(np.int64) - 127)
    else:
        w13 = synth.bf16_expert_weights(E_local, 2 * I, K, seed).float().numpy().astype(np.float64)
        w2 = synth.bf16_expert_weights(E_local, K, I, seed + 1).float().numpy().astype(np.float64)
    return dict(x=x, w13=w13, w2=w2, topk_ids=ids, topk_weights=w.numpy(), E_global=E_global,
                expert_start=expert_start)


@pytest.mark.parametrize("dtype", ["fp8", "mxfp8", "bf16"])
def test_layout_path_equals_per_token_loop(dtype):
    p = small_problem(dtype)
    ref = oracle.forward_per_token(p["x"], p["w13"], p["w2"], p["topk_ids"], p["topk_weights"], dtype,
                                   p["E_global"], p["expert_start"])
    for layout in ("compact", "masked"):
        out = oracle.forward_layout(p["x"], p["w13"], p["w2"], p["topk_ids"], p["topk_weights"], dtype,
                                    p["E_global"], p["expert_start"], layout=layout)
        assert np.array_equal(out, ref), layout
    assert np.count_nonzero(ref) > 0.9 * ref.size


def test_dropped_tokens_give_zero_rows():
    p = small_problem("bf16", E_global=8, E_local=2, expert_start=3)
    out = oracle.forward_layout(p["x"], p["w13"], p["w2"], p["topk_ids"], p["topk_weights"], "bf16",
                                p["E_global"], p["expert_start"])
    ids = p["topk_ids"]
    none_local = ~np.any((ids >= 3) & (ids < 5), axis=1)
    assert none_local.any()
    assert np.all(out[none_local] == 0.0) and np.all(np.any(out[~none_local] != 0, axis=1))


@pytest.mark.parametrize("dtype", ["fp8", "mxfp8", "bf16"])
def test_single_expert_k1_is_textbook_swiglu(dtype):
    rng = np.random.default_rng(2)
    T, K, I = 16, 256, 384
    x = F.bf16_round(rng.standard_normal((T, K)))
    w13 = F.bf16_round(rng.standard_normal((1, 2 * I, K)) * 0.05)
    w2 = F.bf16_round(rng.standard_normal((1, K, I)) * 0.05)
    ids = np.zeros((T, 1), dtype=np.int64)
    wts = np.ones((T, 1), dtype=np.float32)
    out, st = oracle.forward_layout(x, w13, w2, ids, wts, dtype, E_global=1, keep=True)
    a = torch.from_numpy(st["x_in"])
    W1, W3, W2 = (torch.from_numpy(m) for m in (w13[0, :I], w13[0, I:], w2[0]))
    h_ref = torch.nn.functional.silu(a @ W1.T) * (a @ W3.T)
    rows = st["plan"]["src2dst"][:, 0]
    _, inter = oracle.expert_ffn(st["a"][rows], w13[0], w2[0], dtype, keep=True)
    assert torch.allclose(torch.from_numpy(inter["h"]), h_ref, rtol=1e-12, atol=1e-14)
    y_ref = torch.from_numpy(inter["h_in"]) @ W2.T
    assert torch.allclose(torch.from_numpy(inter["y_acc"]), y_ref, rtol=1e-12, atol=1e-14)
    # with weight 1 and a single expert, the layer output is the stored y
    assert np.array_equal(out, F.bf16_round(inter["y_acc"]))


def permutation_expert(K, I, perm1, perm3, perm2, c1, c3, c2):
    """w13 rows: gate n reads x[perm1[n]] * c1, up n reads x[perm3[n]] * c3;
    w2 row m reads h[perm2[m]] * c2 (all entries exact in E4M3 and bf16)."""
    w13 = np.zeros((2 * I, K))
    w13[np.arange(I), perm1] = c1
    w13[I + np.arange(I), perm3] = c3
    w2 = np.zeros((K, I))
    w2[np.arange(K), perm2] = c2
    return w13, w2


def test_hand_computed_permutation_experts():
    """K = I = 128, two experts, values small integers: every intermediate is
    exact, so the expected output is written with math.exp and the bf16
    rounding pinned in test_oracle_formats."""
    K = I = 128
    rng = np.random.default_rng(4)
    p = [rng.permutation(128) for _ in range(6)]
    e0 = permutation_expert(K, I, p[0], p[1], p[2], 1.0, 2.0, 0.5)
    e1 = permutation_expert(K, I, p[3], p[4], p[5], 0.25, 1.0, 1.0)
    w13 = np.stack([e0[0], e1[0]])
    w2 = np.stack([e0[1], e1[1]])
    x = rng.integers(-3, 4, size=(3, K)).astype(np.float64)
    ids = np.array([[0, 1], [1, 0], [1, -1]])
    wts = np.array([[0.75, 0.25], [0.5, 0.5], [1.0, 0.0]], dtype=np.float32)
    out = oracle.forward_layout(x, w13, w2, ids, wts, "bf16", E_global=2)

    def expert(xr, e, c):
        perm1, perm3, perm2 = p[3 * e], p[3 * e + 1], p[3 * e + 2]
        c1, c3, c2 = c
        h = np.array([(xr[perm1[n]] * c1) / (1 + math.exp(-xr[perm1[n]] * c1)) * (xr[perm3[n]] * c3)
                      for n in range(I)])
        h = F.bf16_round(h)
        return F.bf16_round(h[perm2] * c2)

    consts = [(1.0, 2.0, 0.5), (0.25, 1.0, 1.0)]
    for t in range(3):
        acc = np.zeros(K)
        for j in range(2):
            if ids[t, j] >= 0:
                acc += float(wts[t, j]) * expert(x[t], ids[t, j], consts[ids[t, j]])
        assert np.array_equal(out[t], F.bf16_round(acc)), t


def test_dequant_fp8_weights_brute_force():
    """Each element is its E4M3 value times 2^(block exponent) of the 128x128
    block it sits in; checked element by element with plain loops."""
    import math
    rng = np.random.default_rng(6)
    E, N, C = 1, 256, 384
    wb = rng.integers(0, 256, size=(E, N, C), dtype=np.uint8)
    wb[(wb & 0x7F) == 0x7F] = 0x38                          # no NaN codes
    we = rng.integers(-20, 20, size=(E, N // 128, C // 128))
    got = oracle.dequant_fp8_weights(wb, we)
    for n in range(0, N, 7):
        for c in range(0, C, 5):
            b = int(wb[0, n, c])
            sign = -1.0 if b & 0x80 else 1.0
            ef, mf = (b >> 3) & 0xF, b & 7
            v = sign * (mf / 8 * 2.0 ** -6 if ef == 0 else (1 + mf / 8) * 2.0 ** (ef - 7))
            assert got[0, n, c] == v * math.ldexp(1.0, int(we[0, n // 128, c // 128])), (n, c)


@pytest.mark.parametrize("mistake", ["swap_gate_up", "transpose_w2", "drop_combine_term"])
def test_planted_mistakes_are_caught(mistake, monkeypatch):
    """Plant a plausible mistake in the oracle (CPU only) and check that the
    hand-computed pin fails with it."""
    from oracle import moe as om
    if mistake == "swap_gate_up":
        def bad(a, w13_e):
            I = w13_e.shape[0] // 2
            g, u = a @ w13_e[I:].T, a @ w13_e[:I].T
            return g, u, om.silu(g) * u
        monkeypatch.setattr(om, "gemm1_act", bad)
    elif mistake == "transpose_w2":
        monkeypatch.setattr(om, "gemm2", lambda h_in, w2_e: oracle.bf16_round(h_in @ w2_e))

        def bad_ffn(a, w13_e, w2_e, dtype, keep=False):
            g, u, h = om.gemm1_act(a, w13_e)
            h_in, st = om.store_act(h, dtype)
            y = oracle.bf16_round(h_in @ w2_e)
            return (y, {"g": g, "u": u, "h": h, "h_in": h_in, "h_stored": st, "y_acc": h_in @ w2_e}) if keep else y
        monkeypatch.setattr(om, "expert_ffn", bad_ffn)
    else:
        real = om.combine

        def bad(y, src2dst, w):
            s = src2dst.copy()
            s[:, -1] = -1
            return real(y, s, w)
        monkeypatch.setattr(om, "combine", bad)
    with pytest.raises(AssertionError):
        test_hand_computed_permutation_experts()
