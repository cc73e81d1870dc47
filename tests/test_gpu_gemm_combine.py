"""CUDA grouped GEMMs and combine vs the oracle, each fed the CUDA path's own
stage input (so a failure points at one kernel).

Tolerances.  GEMM1: the oracle's fp64 h on the GPU's own dequantised a,
stored the same way (FP8 1x128 UE8M0, MXFP8 1x32 UE8M0 or bf16): relative Frobenius error
<= 2e-3 (FP8 codes may differ by one step where the fp32 and fp64 values of h
straddle a rounding boundary; the flip rate is bounded too).  GEMM2: the
oracle's fp64 y on the GPU's own h, rounded to bf16: <= 2e-3.  Combine: the
oracle's fp64 sum on the GPU's own y: at most one bf16 step per element.
"""

import numpy as np
import pytest
import torch

import oracle
from moe_testlib import Problem, bf16_to_f64, rel_fro

pytestmark = pytest.mark.gpu

CASES = [
    dict(T=128, K=256, I=256, E_global=8, E_local=8, topk=2, dtype="fp8", layout="compact"),
    dict(T=128, K=256, I=256, E_global=8, E_local=8, topk=2, dtype="bf16", layout="compact"),
    dict(T=300, K=640, I=384, E_global=12, E_local=12, topk=4, dtype="fp8", layout="compact", drop_every=5),
    dict(T=300, K=640, I=384, E_global=12, E_local=12, topk=4, dtype="bf16", layout="compact", drop_every=5),
    dict(T=200, K=384, I=256, E_global=64, E_local=16, topk=8, dtype="fp8", layout="masked", expert_start=16),
    dict(T=200, K=384, I=256, E_global=64, E_local=16, topk=8, dtype="bf16", layout="masked", expert_start=16),
    # several 128-row blocks per expert, odd block counts included
    dict(T=700, K=384, I=256, E_global=8, E_local=8, topk=4, dtype="bf16", layout="compact", drop_every=5),
    dict(T=1100, K=256, I=256, E_global=16, E_local=4, topk=4, dtype="bf16", layout="masked", expert_start=4),
    dict(T=700, K=384, I=256, E_global=8, E_local=8, topk=4, dtype="fp8", layout="compact", drop_every=5),
    dict(T=1100, K=256, I=256, E_global=16, E_local=4, topk=4, dtype="fp8", layout="masked", expert_start=4),
    dict(T=700, K=384, I=256, E_global=8, E_local=8, topk=4, dtype="mxfp8", layout="compact", zipf_s=1.2),
    dict(T=600, K=512, I=256, E_global=32, E_local=32, topk=8, dtype="fp8", layout="compact", zipf_s=1.2),
    # masked decode-sized blocks: max_m = 48, one partial block per expert
    dict(T=48, K=384, I=256, E_global=64, E_local=16, topk=8, dtype="fp8", layout="masked", expert_start=16),
    dict(T=48, K=384, I=256, E_global=64, E_local=16, topk=8, dtype="bf16", layout="masked", expert_start=16),
    dict(T=48, K=384, I=256, E_global=64, E_local=16, topk=8, dtype="mxfp8", layout="masked", expert_start=16),
    dict(T=128, K=256, I=256, E_global=8, E_local=8, topk=2, dtype="mxfp8", layout="compact"),
    dict(T=128, K=256, I=256, E_global=8, E_local=8, topk=2, dtype="mxfp4", layout="compact"),
    dict(T=300, K=640, I=384, E_global=12, E_local=12, topk=4, dtype="mxfp4", layout="compact", drop_every=5),
    dict(T=48, K=384, I=256, E_global=64, E_local=16, topk=8, dtype="mxfp4", layout="masked", expert_start=16),
    dict(T=300, K=640, I=384, E_global=12, E_local=12, topk=4, dtype="mxfp8", layout="compact", drop_every=5),
    dict(T=200, K=384, I=256, E_global=64, E_local=16, topk=8, dtype="mxfp8", layout="masked", expert_start=16),
    # masked layouts whose GEMMs run in K segments (GEMM1 4 or 8, GEMM2 2 or 4
    # segments), one of them ragged (5 K blocks in segments of 2 and 3), and
    # experts with rows in two blocks and in several lane quadrants
    dict(T=48, K=1024, I=512, E_global=64, E_local=16, topk=8, dtype="fp8", layout="masked", expert_start=16),
    dict(T=48, K=1024, I=512, E_global=64, E_local=16, topk=8, dtype="bf16", layout="masked", expert_start=16),
    dict(T=100, K=1024, I=512, E_global=64, E_local=16, topk=8, dtype="mxfp8", layout="masked", expert_start=16),
    dict(T=40, K=1024, I=512, E_global=64, E_local=16, topk=8, dtype="mxfp4", layout="masked", expert_start=16),
    dict(T=700, K=640, I=384, E_global=16, E_local=4, topk=4, dtype="fp8", layout="masked", expert_start=4),
]


def _ids(c):
    return "-".join(str(c[k]) for k in ("T", "K", "I", "dtype", "layout"))


def _valid_rows(p, o):
    src = o["src2dst"].reshape(-1)
    return np.sort(src[src >= 0])


def _row_expert(p, o, rows):
    if p.layout == "compact":
        return o["m_indices"][rows]
    return rows // p.max_m


@pytest.mark.parametrize("case", CASES, ids=[_ids(c) for c in CASES])
def test_gemm1_act_matches_oracle(case):
    p = Problem(**case)
    g = p.gpu()
    g.plan(); g.quant(); g.gemm1()
    torch.cuda.synchronize()
    assert g.status() == 0
    o = p.oracle_plan()
    rows = _valid_rows(p, o)
    ex = _row_expert(p, o, rows)
    a = g.decoded("a", rows)
    h_gpu = g.decoded("h", rows)
    h_ref = np.zeros_like(h_gpu)
    for e in np.unique(ex):
        sel = ex == e
        w13, _ = p.expert_weights64(int(e))
        _, _, h = oracle.gemm1_act(a[sel], w13)
        h_ref[sel], _ = oracle.store_act(h, p.dtype)
    err = rel_fro(h_gpu, h_ref)
    assert err <= 2e-3, err
    if p.dtype in ("fp8", "mxfp8", "mxfp4"):
        flips = np.mean(h_gpu != h_ref)
        assert flips <= 5e-3, flips


@pytest.mark.parametrize("case", CASES, ids=[_ids(c) for c in CASES])
def test_gemm2_matches_oracle(case):
    p = Problem(**case)
    g = p.gpu()
    g.plan(); g.quant(); g.gemm1(); g.gemm2()
    torch.cuda.synchronize()
    assert g.status() == 0
    o = p.oracle_plan()
    rows = _valid_rows(p, o)
    ex = _row_expert(p, o, rows)
    h = g.decoded("h", rows)
    y_gpu = bf16_to_f64(g.view("y").index_select(0, torch.as_tensor(rows, device="cuda")))
    y_ref = np.zeros_like(y_gpu)
    for e in np.unique(ex):
        sel = ex == e
        _, w2 = p.expert_weights64(int(e))
        y_ref[sel] = oracle.gemm2(h[sel], w2)
    err = rel_fro(y_gpu, y_ref)
    assert err <= 2e-3, err


COMBINE_CASES = CASES[:6] + CASES[-2:]     # compact and masked, split and unsplit GEMMs


@pytest.mark.parametrize("case", COMBINE_CASES, ids=[_ids(c) for c in COMBINE_CASES])
def test_combine_matches_oracle(case):
    p = Problem(**case)
    g = p.gpu()
    g.plan(); g.quant(); g.gemm1(); g.gemm2(); g.combine()
    torch.cuda.synchronize()
    o = p.oracle_plan()
    y = bf16_to_f64(g.view("y"))
    ref = oracle.combine(y, o["src2dst"], p.w.numpy())
    got = bf16_to_f64(g.out)
    # fp32 accumulation error of the k-term sum, then one bf16 step where the
    # fp32 and fp64 sums straddle a rounding boundary
    mag = np.zeros_like(ref)
    src = o["src2dst"]
    for j in range(p.topk):
        d = src[:, j]
        ok = d >= 0
        mag[ok] += np.abs(p.w.numpy()[ok, j, None]) * np.abs(y[d[ok]])
    _, e = np.frexp(np.maximum(np.abs(ref), 2.0 ** -126))
    bf16_step = np.ldexp(1.0, e - 8)
    bound = bf16_step + 2 * p.topk * 2.0 ** -24 * mag
    assert np.all(np.abs(got - ref) <= bound)
    assert rel_fro(got, ref) <= 1e-3


@pytest.mark.parametrize("layout,I", [("compact", 256), ("masked", 256), ("masked", 512)])
def test_gemm2_block_scales_exact(layout, I):
    """FP8 GEMM2 with every h and w2 element 1.0 (E4M3 0x38): row r of a
    128-row block gets scale 2^(r-64) and weight row block b gets 2^(b%3-1),
    so y[r, n] = I * 2^(r - 64 + b%3 - 1) exactly.  A wrong scale placement
    shows up as the row whose scale was used.  With I = 512 the masked GEMM2
    runs its K loop in two segments, whose exact sums must add up exactly."""
    import moe_expert_layer_ep_gb300 as M
    T, K, E = 256, 384, 2
    kw = dict(T=T, K=K, I=I, E_global=E if layout == "compact" else 4, E_local=E, topk=1, dtype="fp8",
              layout=layout, weight_device="cpu")
    p = Problem(**kw)
    p.ids[:, 0] = torch.arange(T) % E
    p.w2[:] = 0x38
    nb = K // 128
    t_exp = (np.arange(nb) % 3) - 1
    p.w2_sf[:] = torch.as_tensor((t_exp + 127).astype(np.uint8))[None, :, None]
    g = p.gpu()
    g.plan()
    torch.cuda.synchronize()
    o = p.oracle_plan()
    rows = np.sort(o["src2dst"].reshape(-1))
    h = g.view("h")
    h[torch.as_tensor(rows, device="cuda")] = 0x38
    sf = g.view("h_sf")
    r_in = (rows % p.max_m) % 128 if layout == "masked" else rows % 128
    if layout == "masked":
        blk = (rows // p.max_m) * ((p.max_m + 127) // 128) + (rows % p.max_m) // 128
    else:
        blk = rows // 128
    offs = []
    vals = []
    for gidx in range(I // 128):
        offs.append(np.array([M.moe_sf_offset(int(b), gidx, I // 128, int(r)) for b, r in zip(blk, r_in)]))
        vals.append(r_in - 64 + 127)
    offs = np.concatenate(offs)
    vals = np.concatenate(vals).astype(np.uint8)
    sf[torch.as_tensor(offs, device="cuda")] = torch.as_tensor(vals, device="cuda")
    g.gemm2()
    torch.cuda.synchronize()
    assert g.status() == 0
    y = bf16_to_f64(g.view("y").index_select(0, torch.as_tensor(rows, device="cuda")))
    expect = I * np.exp2((r_in - 64)[:, None] + np.repeat(t_exp, 128)[None, :])
    if not np.array_equal(y, expect):
        used = np.log2(np.abs(y[:, 0]) / I) + 64 - t_exp[0]
        bad = np.flatnonzero(y[:, 0] != expect[:, 0])[:8]
        pytest.fail(f"scale placement wrong: row-in-block -> scale row used: "
                    f"{[(int(r_in[i]), float(used[i])) for i in bad]}; col mismatches "
                    f"{np.count_nonzero(y != expect)} of {y.size}")


@pytest.mark.parametrize("layout", ["compact", "masked"])
def test_gemm_stages_full_size_experts(layout):
    """GEMM1 and GEMM2 at the large-prefill shape (K=7168, I=2048, FP8 with
    128x128 weight scales) on every valid row of three experts, each stage fed
    the CUDA path's own input.  Compact: 256 experts with Zipf routing; the
    experts checked are the most used one (several 128-row blocks), the
    highest-numbered one with rows (index above 73: its w13 offset passes 2^31
    elements) and one whose only block is partial.  Masked: 32 local experts
    of 256 at T=256, where the w13 GEMM runs its K loop in segments."""
    import synth
    w = synth.WORKLOADS["fp8_prefill_zipf"]
    if layout == "compact":
        p = Problem(T=1024, K=w["K"], I=w["I"], E_global=256, E_local=256, topk=8, dtype="fp8", layout="compact",
                    seed=w["seed"], zipf_s=w["zipf_s"])
    else:
        p = Problem(T=256, K=w["K"], I=w["I"], E_global=256, E_local=32, topk=8, dtype="fp8", layout="masked",
                    max_m=256, seed=w["seed"] + 5, weight_seed=w["seed"] + 2)
    g = p.gpu()
    g.plan(); g.quant(); g.gemm1(); g.gemm2()
    torch.cuda.synchronize()
    assert g.status() == 0
    o = p.oracle_plan()
    counts = o["counts"]
    nz = np.flatnonzero(counts)
    big = int(nz[np.argmax(counts[nz])])
    high = int(nz.max())
    part = int(next(e for e in nz[np.argsort(counts[nz])] if e not in (big, high)))
    if layout == "compact":
        assert counts[big] > 256 and high > 73 and counts[part] < 128
    else:
        assert g.ctx.ws_layout.k_splits1 > 1 and g.ctx.ws_layout.k_splits2 == 1
    for e in (big, high, part):
        if layout == "compact":
            rows = np.flatnonzero(o["m_indices"] == e)
        else:
            rows = e * p.max_m + np.arange(o["masked_m"][e])
        w13, w2 = p.expert_weights64(e)
        a = g.decoded("a", rows)
        h_gpu = g.decoded("h", rows)
        _, _, h = oracle.gemm1_act(a, w13)
        h_ref, _ = oracle.store_act(h, "fp8")
        assert rel_fro(h_gpu, h_ref) <= 2e-3, (e, "gemm1")
        assert np.mean(h_gpu != h_ref) <= 5e-3, (e, "gemm1 flips")
        y_gpu = bf16_to_f64(g.view("y").index_select(0, torch.as_tensor(rows, device="cuda")))
        assert rel_fro(y_gpu, oracle.gemm2(h_gpu, w2)) <= 2e-3, (e, "gemm2")
