"""Batch invariance (bitwise), device status words and host-side argument
errors of the CUDA path.

Batch invariance follows the method of "[Feature] Support BF16 and
batch-invariant inference with DeepEP v2" (sglang PR #38160 report),
"实现拆解" step 4: a token's output bits must not depend on the batch it is
in, checked with zero tolerance.
"""

import ctypes

import numpy as np
import pytest
import torch

import moe_expert_layer_ep_gb300 as M
import synth
from moe_testlib import Problem

pytestmark = pytest.mark.gpu

K, I, E, TOPK = 7168, 2048, 256, 8
SEED = 0x4D6F45_0003


@pytest.fixture(scope="module")
def weights_fp8():
    w13, w13s = synth.fp8_expert_weights(E, 2 * I, K, SEED + 2, "cuda")
    w2, w2s = synth.fp8_expert_weights(E, K, I, SEED + 3, "cuda")
    return w13, w13s, w2, w2s


@pytest.fixture(scope="module")
def weights_mx():
    w13, w13s = synth.mxfp8_expert_weights(E, 2 * I, K, SEED + 2, "cuda")
    w2, w2s = synth.mxfp8_expert_weights(E, K, I, SEED + 3, "cuda")
    return w13, M.moe_pack_mx_scales(w13s), w2, M.moe_pack_mx_scales(w2s)


@pytest.fixture(scope="module")
def weights_mx4():
    w13, w13s = synth.mxfp4_expert_weights(E, 2 * I, K, SEED + 2, "cuda")
    w2, w2s = synth.mxfp4_expert_weights(E, K, I, SEED + 3, "cuda")
    return w13, M.moe_pack_mx_scales(w13s), w2, M.moe_pack_mx_scales(w2s)


@pytest.fixture(scope="module")
def weights_bf16():
    return synth.bf16_expert_weights(E, 2 * I, K, SEED + 2, "cuda"), synth.bf16_expert_weights(E, K, I, SEED + 3, "cuda")


def _run(dtype, weights, x, ids, w):
    T = x.shape[0]
    shape = M.make_shape(T, K, I, E, E, TOPK, dtype, "compact")
    if dtype in ("fp8", "mxfp8", "mxfp4"):
        ctx = M.moe_ctx_create(shape, weights[0], weights[1], weights[2], weights[3])
    else:
        ctx = M.moe_ctx_create(shape, weights[0], None, weights[1], None)
    ws = M.alloc_workspace(ctx)
    out = torch.empty((T, K), dtype=torch.bfloat16, device="cuda")
    M.moe_forward(ctx, x, ids, w, ws, out)
    torch.cuda.synchronize()
    assert M.moe_read_device_status(ws) == 0
    return out


@pytest.mark.parametrize("dtype", ["fp8", "mxfp8", "mxfp4", "bf16"])
def test_batch_invariance_sweep(dtype, request):
    weights = request.getfixturevalue({"fp8": "weights_fp8", "mxfp8": "weights_mx", "mxfp4": "weights_mx4",
                                       "bf16": "weights_bf16"}[dtype])
    n_probe = 4
    px, pids, pw = synth.probe_tokens(n_probe, K, E, TOPK, SEED, zipf_s=1.2)
    ref = None
    rng = np.random.default_rng(5)
    for T in (1, 7, 128, 1000, 8192):
        for rep in range(2):
            if T == 1:
                rows = []
                for i in range(n_probe):
                    rows.append(_run(dtype, weights, px[i:i + 1].cuda(), pids[i:i + 1].cuda().contiguous(),
                                     pw[i:i + 1].cuda().contiguous())[0].clone())
                got = torch.stack(rows)
            else:
                fx = synth.activations(T, K, 1000 + T + rep, "cuda")
                fids, fw = synth.routing(T, E, TOPK, 2000 + T + rep, zipf_s=1.2)
                pos = rng.choice(T, size=n_probe, replace=False)
                fx[pos] = px.cuda()
                fids[pos] = pids
                fw[pos] = pw
                out = _run(dtype, weights, fx, fids.cuda(), fw.cuda())
                got = out[torch.as_tensor(pos, device="cuda")].clone()
            if ref is None:
                ref = got
            assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), (T, rep)


E_LOCAL_DECODE = 32


def _run_masked(dtype, weights, x, ids, w, max_m):
    """The layer for a rank holding experts 0..31 of 256 (masked layout)."""
    T, EL = x.shape[0], E_LOCAL_DECODE
    shape = M.make_shape(T, K, I, E, EL, TOPK, dtype, "masked", 0, max_m)
    if dtype in ("fp8", "mxfp8", "mxfp4"):
        ctx = M.moe_ctx_create(shape, weights[0][:EL], weights[1][:EL], weights[2][:EL], weights[3][:EL])
    else:
        ctx = M.moe_ctx_create(shape, weights[0][:EL], None, weights[1][:EL], None)
    ws = M.alloc_workspace(ctx)
    out = torch.empty((T, K), dtype=torch.bfloat16, device="cuda")
    M.moe_forward(ctx, x, ids, w, ws, out)
    torch.cuda.synchronize()
    assert M.moe_read_device_status(ws) == 0
    return out, ctx.ws_layout


@pytest.mark.parametrize("dtype", ["fp8", "mxfp8", "mxfp4", "bf16"])
def test_masked_decode_batch_invariance(dtype, request):
    """The masked (expert-parallel decode) layout splits each GEMM tile's K
    loop into segments fixed by K and I alone; a token's output bits must
    still not depend on the batch size, its position or max_m.  Probe tokens
    that route to at least one local expert are placed among filler tokens
    for T = 1, 16, 64 and 256 (max_m = T rounded up to 16), twice each."""
    weights = request.getfixturevalue({"fp8": "weights_fp8", "mxfp8": "weights_mx", "mxfp4": "weights_mx4",
                                       "bf16": "weights_bf16"}[dtype])
    px, pids, pw = synth.probe_tokens(16, K, E, TOPK, SEED + 17)
    local = ((pids >= 0) & (pids < E_LOCAL_DECODE)).any(dim=1).numpy()
    keep = np.flatnonzero(local)[:3]
    assert keep.size == 3
    px, pids, pw = px[keep], pids[keep].contiguous(), pw[keep].contiguous()
    ref = None
    rng = np.random.default_rng(9)
    splits = None
    for T in (1, 16, 64, 256):
        max_m = (T + 15) // 16 * 16
        for rep in range(2):
            if T == 1:
                rows = []
                for i in range(3):
                    out, L = _run_masked(dtype, weights, px[i:i + 1].cuda(), pids[i:i + 1].cuda(),
                                         pw[i:i + 1].cuda(), max_m)
                    rows.append(out[0].clone())
                got = torch.stack(rows)
            else:
                fx = synth.activations(T, K, 3000 + T + rep, "cuda")
                fids, fw = synth.routing(T, E, TOPK, 4000 + T + rep)
                pos = rng.choice(T, size=3, replace=False)
                fx[pos] = px.cuda()
                fids[pos] = pids
                fw[pos] = pw
                out, L = _run_masked(dtype, weights, fx, fids.cuda(), fw.cuda(), max_m)
                got = out[torch.as_tensor(pos, device="cuda")].clone()
            if ref is None:
                ref = got
            assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), (T, rep)
            # the split is the same at every T (it depends on K and I only)
            assert splits in (None, (L.k_splits1, L.k_splits2))
            splits = (L.k_splits1, L.k_splits2)
    assert splits[0] > 1 and splits[1] == 1      # K=7168, I=2048: w13 in segments, w2 whole
    assert ref.abs().max() > 0


def test_bad_expert_id_sets_status_and_is_dropped():
    p = Problem(T=64, K=256, I=128, E_global=8, E_local=8, topk=2, dtype="fp8", layout="compact",
                weight_device="cpu")
    p.ids[3, 1] = 9
    p.ids[5, 0] = -5
    g = p.gpu()
    g.forward()
    assert g.status() == M.STATUS["MOE_ERR_EXPERT_ID"]
    src = g.view("src2dst").cpu().numpy().reshape(64, 2)
    assert src[3, 1] == -1 and src[5, 0] == -1 and np.all(src[0] >= 0)


def test_masked_overflow_sets_status():
    p = Problem(T=4, K=256, I=128, E_global=16, E_local=4, topk=2, dtype="fp8", layout="masked", max_m=4,
                weight_device="cpu")
    p.ids[:] = 1          # duplicate ids in every row: expert 1 gets 8 > max_m assignments
    g = p.gpu()
    g.forward()
    assert g.status() == M.STATUS["MOE_ERR_MASKED_OVERFLOW"]
    assert g.view("masked_m").cpu().numpy()[1] == 4


def test_kernel_wait_timeout_is_reported_not_hung():
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    M.moe_selftest_wait_timeout(ws, 2_000_000)        # 2 ms limit, nothing ever arrives
    assert M.moe_read_device_status(ws) == M.STATUS["MOE_ERR_TIMEOUT"]
    # the context is still usable afterwards
    p = Problem(T=16, K=256, I=128, E_global=8, E_local=8, topk=2, dtype="bf16", layout="compact",
                weight_device="cpu")
    g = p.gpu()
    g.forward()
    assert g.status() == 0


def test_host_side_errors():
    p = Problem(T=16, K=256, I=128, E_global=8, E_local=8, topk=2, dtype="fp8", layout="compact",
                weight_device="cuda")
    good = M.make_shape(16, 256, 128, 8, 8, 2, "fp8", "compact")
    handle = ctypes.c_void_p()
    bad_k = M.make_shape(16, 200, 128, 8, 8, 2, "fp8", "compact")
    code = M._lib.moe_ctx_create(ctypes.byref(bad_k), p.w13.data_ptr(), p.w13_sf.data_ptr(), p.w2.data_ptr(),
                                 p.w2_sf.data_ptr(), ctypes.byref(handle))
    assert code == M.STATUS["MOE_ERR_UNSUPPORTED"]
    bad_align = M._lib.moe_ctx_create(ctypes.byref(good), p.w13.data_ptr() + 8, p.w13_sf.data_ptr(),
                                      p.w2.data_ptr(), p.w2_sf.data_ptr(), ctypes.byref(handle))
    assert bad_align == M.STATUS["MOE_ERR_MISALIGNED"]
    code = M._lib.moe_ctx_create(ctypes.byref(good), p.w13.data_ptr(), None, p.w2.data_ptr(),
                                 p.w2_sf.data_ptr(), ctypes.byref(handle))
    assert code == M.STATUS["MOE_ERR_DTYPE_MISMATCH"]
    ctx = M.moe_ctx_create(good, p.w13, p.w13_sf, p.w2, p.w2_sf)
    ws = M.alloc_workspace(ctx)
    ids = p.ids.cuda()
    code = M._lib.moe_plan_layout(ctx.handle, ids.data_ptr() + 4, ws.data_ptr(), M._stream(None))
    assert code == M.STATUS["MOE_ERR_MISALIGNED"]
    code = M._lib.moe_plan_layout(ctx.handle, ids.data_ptr(), ws.data_ptr() + 16, M._stream(None))
    assert code == M.STATUS["MOE_ERR_MISALIGNED"]
    bad_masked = M.make_shape(16, 256, 128, 64, 8, 2, "fp8", "masked", max_m=8)
    with pytest.raises(M.MoeError) as e:
        M.moe_ctx_create(bad_masked, p.w13, p.w13_sf, p.w2, p.w2_sf)
    assert e.value.code == M.STATUS["MOE_ERR_INVALID_ARG"]
