"""The no-allocation layout entry point (moe_plan_layout_noalloc).

Some callers cannot allocate device memory: code inside a framework whose
memory planner owns the device heap and hands it only the tensors it reads
and writes.  For them the layout step keeps its scratch in a fixed array in
the library's device image and takes caller-owned output buffers.  This test
calls it through the C-ABI twice in a row, with different routings, and
checks every output against the workspace-based moe_plan_layout on the same
inputs; the layout is integer work, so the comparison is exact.  It also
checks the size limit is reported as an error.

This file is collected last on purpose: it must pass alone in a fresh process
and after the other tests, and a failure here leaves the rest of a run that
stops at the first failure already done.
"""

import numpy as np
import pytest
import torch

import moe_expert_layer_ep_gb300 as M
import synth

pytestmark = pytest.mark.gpu

KEYS_COMMON = ("status", "meta", "counts", "src2dst", "block_info")
KEYS_COMPACT = ("padded", "start", "m_indices")
KEYS_MASKED = ("masked_m",)


def _reference(shape, ids):
    """moe_plan_layout through a context and workspace (tiny dummy weights:
    the layout does not read them)."""
    E, K, I = shape.E_local, shape.K, shape.I
    w13 = torch.zeros((E, 2 * I, K), dtype=torch.uint8, device="cuda")
    w2 = torch.zeros((E, K, I), dtype=torch.uint8, device="cuda")
    w13s = torch.full((E, 2 * I // 128, K // 128), 127, dtype=torch.uint8, device="cuda")
    w2s = torch.full((E, K // 128, I // 128), 127, dtype=torch.uint8, device="cuda")
    ctx = M.moe_ctx_create(shape, w13, w13s, w2, w2s)
    ws = M.alloc_workspace(ctx)
    M.moe_plan_layout(ctx, ids, ws)
    torch.cuda.synchronize()
    keys = KEYS_COMMON + (KEYS_MASKED if ctx.masked else KEYS_COMPACT)
    return {k: M.ws_view(ctx, ws, k).clone() for k in keys}, ctx.ws_layout


def _outputs_like(ref):
    return {k: torch.full_like(v, -7) for k, v in ref.items()}


# (layout, T, E_global, E_local, expert_start, topk, Zipf exponent).  The
# one-CTA plan serves up to 2048 assignments; the three-kernel plan, which
# uses the static scratch array, serves larger problems, so the compact case
# and the second masked case take that path.
CASES = [("compact", 8192, 256, 256, 0, 8, 1.2),
         ("masked", 256, 256, 32, 32, 8, None),
         ("masked", 1024, 256, 32, 32, 8, None)]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}-T{c[1]}" for c in CASES])
def test_noalloc_plan_matches_workspace_plan_twice(case):
    layout, T, E_global, E_local, start, topk, zipf = case
    shape = M.make_shape(T, 128, 128, E_global, E_local, topk, "fp8", layout, expert_start=start,
                         max_m=T if layout == "masked" else 0)
    for call in range(2):
        ids, _ = synth.routing(T, E_global, topk, 100 + call, zipf)
        ids = ids.cuda()
        ref, _ = _reference(shape, ids)
        out = _outputs_like(ref)
        M.moe_plan_layout_noalloc(shape, ids, out)
        torch.cuda.synchronize()
        # meta[0:2] and the first meta[1] block-table entries are defined;
        # everything else listed is written in full
        nblk = int(ref["meta"][1].item())
        assert torch.equal(out["meta"][:2], ref["meta"][:2]), call
        assert torch.equal(out["block_info"][:4 * nblk], ref["block_info"][:4 * nblk]), call
        for k in ref:
            if k not in ("meta", "block_info"):
                assert torch.equal(out[k], ref[k]), (call, k)
        assert out["status"][0].item() == 0 and nblk > 0


def test_noalloc_plan_rejects_problems_beyond_its_scratch():
    T, E, topk = 65536, 256, 8          # 2048 chunks * 256 experts + 524288 > 262144 words
    shape = M.make_shape(T, 128, 128, E, E, topk, "fp8", "compact")
    ids = torch.zeros((T, topk), dtype=torch.int32, device="cuda")
    with pytest.raises(M.MoeError) as e:
        M.moe_plan_layout_noalloc(shape, ids, {"status": ids, "meta": ids, "counts": ids, "src2dst": ids,
                                               "block_info": ids, "padded": ids, "start": ids,
                                               "m_indices": ids})
    assert e.value.code == M.STATUS["MOE_ERR_BUFFER_TOO_SMALL"]
