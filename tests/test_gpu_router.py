"""CUDA fp32 router vs the oracle.

Logits: against fp64 within 2^-24 * K * sum|x w| -- the bound of a K-term
sequential fp32 sum, which also covers the tensor-core path (exact products,
3K/16 + 16 fp32 accumulations of at most 2^-23 relative error each, then
the segment fold).  Top-k ids:
bit-exact against the oracle's selection applied to the kernel's own fp32
logits (the comparison that decides an id is taken in the kernel's
precision), including rows with tied logits.  Weights: the oracle's softmax
of the same logits, within a few fp32 ulps.  Batch invariance: a token's
outputs do not depend on the batch around it, whichever kernel its batch
size selects: a large batch adds each tile's K segments inside the logits
kernel, a small one through a partial buffer, in the same order.
"""

import numpy as np
import pytest
import torch

import moe_expert_layer_ep_gb300 as M
from oracle import router as R

pytestmark = pytest.mark.gpu


def _inputs(T, K, E, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((T, K), generator=g).to(torch.bfloat16)
    w = (torch.randn((E, K), generator=g) * 0.02).float()
    return x, w


def _planes(w):
    return M.moe_router_prepare(w.cuda())


def _check(x, w, topk, rows=None):
    ids, wts, z = M.moe_route(x.cuda(), _planes(w), topk)
    torch.cuda.synchronize()
    z = z.cpu().numpy()
    ids = ids.cpu().numpy()
    wts = wts.cpu().numpy()
    rows = np.arange(x.shape[0]) if rows is None else np.asarray(rows)
    x64 = x.float().numpy().astype(np.float64)[rows]
    w64 = w.numpy().astype(np.float64)
    ref_z = R.logits(x64, w64)
    bound = 2.0 ** -24 * x.shape[1] * (np.abs(x64) @ np.abs(w64).T) + 1e-30
    assert np.all(np.abs(z[rows] - ref_z) <= bound)
    ref_ids = R.select_topk(z[rows], topk)
    assert np.array_equal(ids[rows], ref_ids)
    ref_w = R.topk_softmax(z[rows].astype(np.float64), ref_ids)
    assert np.allclose(wts[rows], ref_w, rtol=4e-6, atol=1e-7)
    return ids, wts, z


@pytest.mark.parametrize("T,K,E,topk", [(1, 256, 8, 2), (77, 512, 64, 8), (300, 2048, 128, 8), (129, 7168, 256, 8),
                                        (257, 1024, 40, 4), (5, 1024, 1000, 64), (64, 1152, 37, 6),
                                        (1, 7168, 256, 8), (700, 384, 300, 33)])
def test_router_matches_oracle(T, K, E, topk):
    x, w = _inputs(T, K, E, T + E)
    _check(x, w, topk)


def test_router_ties_go_to_lower_id():
    x, w = _inputs(50, 256, 32, 3)
    w[7] = w[3]            # identical rows: identical logits, bit for bit
    w[20] = w[3]
    w[31] = w[30]
    ids, _, z = _check(x, w, 8)
    assert np.array_equal(z[:, 7], z[:, 3]) and np.array_equal(z[:, 20], z[:, 3])
    for t in range(50):
        row = ids[t].tolist()
        if 3 in row and 7 in row:
            assert row.index(3) < row.index(7) < (row.index(20) if 20 in row else 99)


def test_router_full_size_sampled_and_batch_invariant():
    T, K, E = 8192, 7168, 256
    x, w = _inputs(T, K, E, 11)
    ids, wts, z = _check(x, w, 8, rows=[0, 1, 4095, 8191])
    # the same tokens routed in a batch of 7 give the same bits
    sub = torch.cat([x[4095:4096], x[:3], x[8191:8192], x[1:4]])
    ids2, wts2, z2 = M.moe_route(sub.cuda(), _planes(w), 8)
    torch.cuda.synchronize()
    assert np.array_equal(z2.cpu().numpy()[0], z[4095]) and np.array_equal(z2.cpu().numpy()[4], z[8191])
    assert np.array_equal(ids2.cpu().numpy()[1:4], ids[:3]) and np.array_equal(wts2.cpu().numpy()[4], wts[8191])


def test_router_logits_identical_across_batch_sizes():
    """Batches of 1, 40, 256 and 300 tokens cover one to three token tiles
    and a ragged K segment; every token's logits, ids and weights are the
    same bits."""
    x, w = _inputs(300, 1152, 37, 5)
    wc = _planes(w)
    full = [t.cpu() for t in M.moe_route(x.cuda(), wc, 6)]
    for n in (1, 40, 256):
        part = [t.cpu() for t in M.moe_route(x[:n].cuda(), wc, 6)]
        for a, b in zip(part, full):
            assert torch.equal(a, b[:n])


def test_router_folded_and_partial_paths_agree_bitwise():
    """A batch whose 128 x 128 tiles fill most of the GPU is folded inside
    the logits kernel, a smaller one through the partial buffer: the same
    tokens get the same bits either way (K = 1152 ends in a short segment)."""
    x, w = _inputs(2048, 1152, 1024, 21)      # 16 x 8 = 128 tiles
    wc = _planes(w)
    big = [t.cpu() for t in M.moe_route(x.cuda(), wc, 8)]
    rows = [0, 5, 517, 2047]
    small = [t.cpu() for t in M.moe_route(x[rows].cuda(), wc, 8)]
    for a, b in zip(small, big):
        assert torch.equal(a, b[rows])
    _check(x[:200], w, 8)


def test_router_weight_split_is_exact():
    """plane0 + plane1 + plane2 == w exactly, for normal-range weights of
    many magnitudes (the sum is formed in fp64, where it is exact)."""
    g = torch.Generator().manual_seed(9)
    w = torch.randn((64, 1024), generator=g) * torch.exp2(torch.randint(-60, 60, (64, 1), generator=g).float())
    w[0, :8] = torch.tensor([1.0, -1.0, 3.0e38, -2.0 ** -100, 1.0 + 2.0 ** -23, 0.0, -0.0, 2.0 ** -110])
    planes = M.moe_router_prepare(w.cuda()).cpu().float().double()
    assert torch.equal(planes.sum(0), w.double())


def test_router_host_errors():
    x = torch.zeros((4, 256), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((8, 100), dtype=torch.float32, device="cuda")
    with pytest.raises(M.MoeError) as e:
        M.moe_router_prepare(w)
    assert e.value.code == M.STATUS["MOE_ERR_UNSUPPORTED"]
    planes = M.moe_router_prepare(torch.zeros((8, 256), dtype=torch.float32, device="cuda"))
    small = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(M.MoeError) as e:
        M.moe_route(x, planes, 2, ws=small)
    assert e.value.code == M.STATUS["MOE_ERR_BUFFER_TOO_SMALL"]
