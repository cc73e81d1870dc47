"""CUDA plan + quant-scatter vs the oracle: bit-exact (integer layout, FP8
bytes, UE8M0 exponents)."""

import numpy as np
import pytest
import torch

import oracle
from moe_testlib import Problem

pytestmark = pytest.mark.gpu

CASES = [
    # T, K, I, E_global, E_local, topk, dtype, layout, expert_start, zipf, drop
    dict(T=128, K=256, I=256, E_global=8, E_local=8, topk=2, dtype="fp8", layout="compact"),
    dict(T=300, K=512, I=256, E_global=16, E_local=16, topk=4, dtype="fp8", layout="compact", drop_every=5),
    dict(T=300, K=384, I=128, E_global=24, E_local=10, topk=6, dtype="bf16", layout="compact", expert_start=7,
         drop_every=3),
    dict(T=1, K=256, I=128, E_global=64, E_local=16, topk=8, dtype="fp8", layout="masked"),
    dict(T=77, K=256, I=128, E_global=64, E_local=32, topk=8, dtype="fp8", layout="masked", expert_start=32),
    dict(T=2000, K=256, I=128, E_global=256, E_local=256, topk=8, dtype="bf16", layout="compact", zipf_s=1.2),
    dict(T=8192, K=128, I=128, E_global=256, E_local=256, topk=8, dtype="fp8", layout="compact", zipf_s=1.2),
    dict(T=0, K=256, I=128, E_global=8, E_local=8, topk=2, dtype="fp8", layout="compact"),
    dict(T=300, K=2304, I=128, E_global=16, E_local=16, topk=4, dtype="mxfp8", layout="compact", drop_every=5),
    dict(T=77, K=384, I=128, E_global=64, E_local=32, topk=8, dtype="mxfp8", layout="masked", expert_start=32),
    dict(T=65, K=512, I=128, E_global=16, E_local=16, topk=4, dtype="mxfp4", layout="compact"),
]


def _ids(c):
    return "-".join(f"{k}{v}" for k, v in c.items() if k in ("T", "dtype", "layout", "E_local"))


@pytest.mark.parametrize("case", CASES, ids=[_ids(c) for c in CASES])
def test_plan_matches_oracle_bit_exact(case):
    p = Problem(**case, weight_device="cpu")
    g = p.gpu()
    g.plan()
    torch.cuda.synchronize()
    o = p.oracle_plan()
    assert g.status() == 0
    assert np.array_equal(g.view("counts").cpu().numpy(), o["counts"])
    assert np.array_equal(g.view("src2dst").cpu().numpy().reshape(p.T, p.topk), o["src2dst"])
    meta = g.view("meta").cpu().numpy()
    bi = g.view("block_info").cpu().numpy().reshape(-1, 4)
    if p.layout == "compact":
        assert np.array_equal(g.view("padded").cpu().numpy(), o["padded"])
        assert np.array_equal(g.view("start").cpu().numpy(), o["start"])
        assert np.array_equal(g.view("m_indices").cpu().numpy(), o["m_indices"])
        assert meta[0] == o["padded"].sum() and meta[1] == o["padded"].sum() // 128
        # block table: expert of each block and its valid rows, from m_indices
        mi = o["m_indices"]
        for j in range(meta[1]):
            rows = mi[j * 128:(j + 1) * 128]
            assert bi[j, 0] == rows[0] and bi[j, 1] == j * 128 and bi[j, 3] == np.count_nonzero(rows >= 0)
    else:
        mm = o["masked_m"]
        assert np.array_equal(g.view("masked_m").cpu().numpy(), mm)
        nblk = (mm + 127) // 128
        assert meta[1] == nblk.sum()
        j = 0
        for e in range(p.E_local):
            for b in range(nblk[e]):
                assert tuple(bi[j]) == (e, e * p.max_m + 128 * b, 128 * b, min(128, mm[e] - 128 * b))
                j += 1


@pytest.mark.parametrize("case", CASES, ids=[_ids(c) for c in CASES])
def test_quant_scatter_matches_oracle_bit_exact(case):
    p = Problem(**case, weight_device="cpu")
    g = p.gpu()
    g.plan()
    g.quant()
    torch.cuda.synchronize()
    o = p.oracle_plan()
    src = o["src2dst"].reshape(-1)
    tok = np.repeat(np.arange(p.T), p.topk)
    keep = src >= 0
    rows, toks = src[keep], tok[keep]
    if rows.size == 0:
        return
    a = g.view("a")
    got = a.index_select(0, torch.as_tensor(rows, device=a.device)).cpu()
    x64 = p.x64()
    if p.dtype in ("fp8", "mxfp8", "mxfp4"):   # MXFP4 weights keep MXFP8 activations
        q, s = oracle.quant_fp8_1x128(x64) if p.dtype == "fp8" else oracle.quant_mxfp8_1x32(x64)
        assert np.array_equal(got.numpy(), oracle.e4m3_bits(q)[toks])
        assert np.array_equal(g.sf_bytes("a_sf", rows), (s + 127).astype(np.uint8)[toks])
    else:
        assert torch.equal(got.view(torch.int16), p.x[toks].view(torch.int16))


def test_quant_edge_values_fp8():
    """Zero groups, subnormal-bf16 groups, exact power-of-two boundaries and
    values that round to the saturation boundary."""
    p = Problem(T=6, K=512, I=128, E_global=4, E_local=4, topk=1, dtype="fp8", layout="compact",
                weight_device="cpu")
    x = torch.randn((6, 512), dtype=torch.float32)
    x[0, :128] = 0.0
    x[1, 128:256] = 1e-39                          # bf16 subnormals
    x[2, :128] = 448.0 * 4                         # amax exactly 448 * 2^2
    x[3, :128] = torch.linspace(-3.0, 3.0, 128)
    x[4, 256:384] = 3.0e38                          # near bf16 max
    x[5] = -0.0
    p.x = x.to(torch.bfloat16)
    g = p.gpu()
    g.plan()
    g.quant()
    torch.cuda.synchronize()
    o = p.oracle_plan()
    rows = o["src2dst"][:, 0]
    q, s = oracle.quant_fp8_1x128(p.x64())
    got = g.view("a").index_select(0, torch.as_tensor(rows, device="cuda")).cpu().numpy()
    assert np.array_equal(got, oracle.e4m3_bits(q))
    assert np.array_equal(g.sf_bytes("a_sf", rows), (s + 127).astype(np.uint8))


SMALL_FORWARD_CASES = [c for c in CASES if 0 < c["T"] * c["topk"] <= 2048 and c["E_local"] <= 256]


@pytest.mark.parametrize("case", SMALL_FORWARD_CASES, ids=[_ids(c) for c in SMALL_FORWARD_CASES])
def test_forward_quant_destinations_match_the_plan(case):
    """Inside moe_forward, small problems plan and quantise in one launch,
    the quantising CTAs forming their destination rows from the routing
    (beside the planning CTA, not after it).  The expert rows and scales
    must be the bytes the plan-driven moe_quant_scatter writes, and src2dst
    the plan's."""
    p = Problem(**case, weight_device="cpu")
    ref = p.gpu()
    ref.plan()
    ref.quant()
    torch.cuda.synchronize()
    fwd = p.gpu()
    fwd.forward()
    torch.cuda.synchronize()
    assert fwd.status() == 0
    src = ref.view("src2dst").cpu().numpy()
    assert np.array_equal(fwd.view("src2dst").cpu().numpy(), src)
    rows = np.sort(src[src >= 0])
    if rows.size == 0:
        return
    idx = torch.as_tensor(rows, device="cuda")
    a_ref, a_fwd = ref.view("a").index_select(0, idx), fwd.view("a").index_select(0, idx)
    if p.dtype == "bf16":
        assert torch.equal(a_ref.view(torch.int16), a_fwd.view(torch.int16))
    else:
        assert torch.equal(a_ref, a_fwd)
        assert np.array_equal(ref.sf_bytes("a_sf", rows), fwd.sf_bytes("a_sf", rows))
