"""MXFP8-specific checks of the CUDA path (the general parity suites carry
MXFP8 cases too):

* moe_pack_mx_scales writes the documented chunk order, bit for bit;
* GEMM2 with every h and w2 element 1.0 and power-of-two scales that differ
  per row and per 32-column block: the fp32 sum is exact (eight terms
  32 * 2^a with |a| <= 6 span at most 20 bits), so y is exactly its bf16
  rounding, and a scale byte read for the wrong row, the wrong 32-column
  block or the wrong weight row changes the result.
"""

import ctypes

import numpy as np
import pytest
import torch

import moe_expert_layer_ep_gb300 as M
import oracle
from moe_testlib import Problem, bf16_to_f64

pytestmark = pytest.mark.gpu


def test_pack_mx_scales_layout():
    E, N, C = 2, 256, 640
    src = torch.randint(0, 256, (E, N, C // 32), dtype=torch.uint8)
    got = M.moe_pack_mx_scales(src.cuda()).cpu().numpy().reshape(-1)
    s = src.numpy()
    want = np.zeros(E * N * C // 32, dtype=np.uint8)
    for e in range(E):
        for n in range(N):
            for blk in range(C // 32):
                kg, c = blk // 4, blk % 4
                chunk = (e * (N // 128) + n // 128) * (C // 128) + kg
                r = n % 128
                want[chunk * 512 + 16 * (r % 32) + 4 * (r // 32) + c] = s[e, n, blk]
    assert np.array_equal(got, want)


def test_pack_mx_scales_padded_rows():
    """Scale rows padded to 32 bytes (C/32 = 20 used) pack like unpadded ones."""
    E, N, C = 2, 128, 640
    src = torch.randint(0, 256, (E, N, C // 32), dtype=torch.uint8)
    padded = torch.randint(0, 256, (E, N, 32), dtype=torch.uint8)
    padded[:, :, :C // 32] = src
    a = M.moe_pack_mx_scales(src.cuda()).cpu()
    b = M.moe_pack_mx_scales(padded.cuda(), C=C).cpu()
    assert torch.equal(a, b)


def test_pack_mx_scales_host_errors():
    a = torch.zeros(2 * 128 * 4, dtype=torch.uint8, device="cuda")
    with pytest.raises(M.MoeError) as e:
        M.moe_pack_mx_scales(a.view(2, 128, 4), out=a.view(2, 128, 4))   # in place: overlap
    assert e.value.code == M.STATUS["MOE_ERR_INVALID_ARG"]


@pytest.mark.parametrize("layout", ["compact", "masked"])
def test_gemm2_mx_scales_exact(layout):
    T, K, I, E = 256, 384, 256, 2
    kw = dict(T=T, K=K, I=I, E_global=E if layout == "compact" else 4, E_local=E, topk=1, dtype="mxfp8",
              layout=layout, weight_device="cpu")
    p = Problem(**kw)
    p.ids[:, 0] = torch.arange(T) % E
    p.w2[:] = 0x38                                            # every weight element 1.0
    rng = np.random.default_rng(7)
    sw = rng.integers(-3, 4, size=(E, K, I // 32))            # weight row n, block c exponent
    p.w2_sf[:] = torch.as_tensor((sw + 127).astype(np.uint8))
    g = p.gpu()
    g.plan()
    torch.cuda.synchronize()
    o = p.oracle_plan()
    rows = np.sort(o["src2dst"].reshape(-1))
    expert = (rows // p.max_m) if layout == "masked" else o["m_indices"][rows]
    h = g.view("h")
    h[torch.as_tensor(rows, device="cuda")] = 0x38           # every h element 1.0
    sh = rng.integers(-3, 4, size=(len(rows), I // 32))       # h row, block c exponent
    r_in = (rows % p.max_m) % 128 if layout == "masked" else rows % 128
    if layout == "masked":
        blk = (rows // p.max_m) * ((p.max_m + 127) // 128) + (rows % p.max_m) // 128
    else:
        blk = rows // 128
    sf = g.view("h_sf")
    for c in range(I // 32):
        off = (blk * (I // 128) + c // 4) * 512 + 16 * (r_in % 32) + 4 * (r_in // 32) + c % 4
        sf[torch.as_tensor(off, device="cuda")] = torch.as_tensor((sh[:, c] + 127).astype(np.uint8), device="cuda")
    g.gemm2()
    torch.cuda.synchronize()
    assert g.status() == 0
    y = bf16_to_f64(g.view("y").index_select(0, torch.as_tensor(rows, device="cuda")))
    # y[row, n] = sum_c 32 * 2^(sh[row, c] + sw[e, n, c])
    expect = oracle.bf16_round(32.0 * np.einsum("rc,rnc->rn", np.exp2(sh), np.exp2(sw[expert])))
    assert np.array_equal(y, expect), np.count_nonzero(y != expect)


def test_mxfp4_weights_need_32_byte_alignment():
    # packed E2M1 weights are read by TMA copies that require 32-byte-aligned
    # bases; a 16-byte-aligned pointer is rejected at context creation
    p = Problem(T=16, K=256, I=128, E_global=8, E_local=8, topk=2, dtype="mxfp4", layout="compact",
                weight_device="cuda")
    g = p.gpu()   # packs the scales as the context expects them
    shape = M.make_shape(16, 256, 128, 8, 8, 2, "mxfp4", "compact")
    handle = ctypes.c_void_p()
    for w13_off, w2_off in ((16, 0), (0, 16)):
        code = M._lib.moe_ctx_create(ctypes.byref(shape), g.w13.data_ptr() + w13_off, g.w13_sf.data_ptr(),
                                     g.w2.data_ptr() + w2_off, g.w2_sf.data_ptr(), ctypes.byref(handle))
        assert code == M.STATUS["MOE_ERR_MISALIGNED"]
