"""CUDA load-time UE8M0 requantisation vs the oracle: bit-exact bytes and
exponents; in-place operation; a full-size expert slice of the large
prefill's w13."""

import numpy as np
import pytest
import torch

import moe_expert_layer_ep_gb300 as M
from oracle import requant as RQ

pytestmark = pytest.mark.gpu


def _case(E, N, C, seed):
    g = torch.Generator().manual_seed(seed)
    w = torch.randint(0, 256, (E, N, C), generator=g, dtype=torch.int32).to(torch.uint8)
    w[(w & 0x7F) == 0x7F] = 0x3A
    nb = (E, N // 128, C // 128)
    s = (torch.rand(nb, generator=g) + 1.0) * torch.exp2(torch.randint(-14, -8, nb, generator=g).float())
    return w, s.float()


@pytest.mark.parametrize("E,N,C", [(3, 256, 384), (1, 128, 128), (2, 512, 1024)])
def test_requant_bit_exact(E, N, C):
    w, s = _case(E, N, C, 7 + E)
    s[0, 0, 0] = 0.0                                 # an all-zero block
    ref_w, ref_e = RQ.requant_block_ue8m0(w.numpy(), s.numpy())
    out_w, out_s = M.moe_requant_weights_ue8m0(w.cuda(), s.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(out_w.cpu().numpy(), ref_w)
    assert np.array_equal(out_s.cpu().numpy().astype(np.int64) - 127, ref_e)


def test_requant_signed_and_extreme_scales_bit_exact():
    """Negative scales (the block maximum is taken over |v|), zero, scales
    whose products fall below the fp32 normal range (exponent clamped at
    -127) and scales whose products approach the fp32 maximum."""
    w, s = _case(2, 256, 512, 23)
    s = s.clone()
    s[0, 0, :] = -s[0, 0, :]
    s[0, 1, 0] = -0.0
    s[1, 0, 0] = 2.0 ** -140                         # products below the fp32 normal range
    s[1, 0, 1] = 2.0 ** 100                          # large exponents (finite products)
    s[1, 1, 2] = -(2.0 ** -100)
    s[1, 1, 3] = 3.0e38 / 448.0
    ref_w, ref_e = RQ.requant_block_ue8m0(w.numpy(), s.numpy())
    out_w, out_s = M.moe_requant_weights_ue8m0(w.cuda(), s.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(out_w.cpu().numpy(), ref_w)
    assert np.array_equal(out_s.cpu().numpy().astype(np.int64) - 127, ref_e)


def test_requant_in_place_matches():
    w, s = _case(2, 256, 256, 3)
    a = w.cuda()
    ref_w, ref_s = M.moe_requant_weights_ue8m0(a, s.cuda())
    b = w.cuda()
    M.moe_requant_weights_ue8m0(b, s.cuda(), w_out=b)
    torch.cuda.synchronize()
    assert torch.equal(a, w.cuda()) and torch.equal(b, ref_w)


def test_requant_full_size_expert_slice():
    """One expert of the large-prefill w13 ([4096, 7168]) against the oracle."""
    w, s = _case(1, 4096, 7168, 11)
    ref_w, ref_e = RQ.requant_block_ue8m0(w.numpy(), s.numpy())
    out_w, out_s = M.moe_requant_weights_ue8m0(w.cuda(), s.cuda())
    assert np.array_equal(out_w.cpu().numpy(), ref_w)
    assert np.array_equal(out_s.cpu().numpy().astype(np.int64) - 127, ref_e)


def test_requant_host_errors():
    w = torch.zeros((1, 128, 100), dtype=torch.uint8, device="cuda")
    s = torch.ones((1, 1, 1), dtype=torch.float32, device="cuda")
    code = M._lib.moe_requant_weights_ue8m0(w.data_ptr(), s.data_ptr(), w.data_ptr(), s.data_ptr(), 1, 128, 100,
                                            M._stream(None))
    assert code == M.STATUS["MOE_ERR_UNSUPPORTED"]
