"""Seeded random shapes through the whole layer against the oracle: odd
token counts, K / I multiples of 128 that are not multiples of 256, expert
ranges with an offset, dropped ids, every dtype and both layouts.  The bar is
the end-to-end one: relative Frobenius error <= 2e-3, and rows without a
local assignment exactly zero."""

import numpy as np
import pytest

from moe_testlib import Problem, bf16_to_f64, rel_fro

pytestmark = pytest.mark.gpu


def _case(seed):
    rng = np.random.default_rng(1000 + seed)
    E_global = int(rng.integers(2, 65))
    E_local = int(rng.integers(1, E_global + 1))
    expert_start = int(rng.integers(0, E_global - E_local + 1))
    T = int(rng.integers(1, 401))
    layout = "masked" if rng.random() < 0.4 else "compact"
    return dict(T=T, K=128 * int(rng.integers(1, 9)), I=128 * int(rng.integers(1, 7)), E_global=E_global,
                E_local=E_local, expert_start=expert_start, topk=int(rng.integers(1, min(8, E_global) + 1)),
                dtype=["fp8", "mxfp8", "mxfp4", "bf16"][seed % 4], layout=layout,
                max_m=T + int(rng.integers(0, 20)) if layout == "masked" else 0,
                drop_every=int(rng.integers(0, 6)), seed=seed)


@pytest.mark.parametrize("seed", range(24))
def test_random_shapes_match_oracle(seed):
    case = _case(seed)
    p = Problem(**case)
    g = p.gpu()
    out = bf16_to_f64(g.forward())
    assert g.status() == 0, case
    ref = p.oracle_forward()
    assert rel_fro(out, ref) <= 2e-3, case
    ids = p.ids.numpy()
    local = (ids >= p.expert_start) & (ids < p.expert_start + p.E_local)
    assert np.all(out[~local.any(axis=1)] == 0.0), case


@pytest.mark.parametrize("case", [dict(T=96, K=128 * 136, I=256, E_global=4, E_local=4, topk=2, layout="compact"),
                                  dict(T=96, K=256, I=128 * 136, E_global=4, E_local=4, topk=2, layout="compact"),
                                  dict(T=40, K=128 * 136, I=256, E_global=8, E_local=4, topk=2, layout="masked")],
                         ids=["long-K-gemm1", "long-K-gemm2", "long-K-masked"])
def test_reductions_longer_than_128_K_blocks(case):
    """FP8 reductions of 136 K blocks (K or I = 17408): the weight-scale warp
    holds the scale words of 32 four-block quads at a time and must fetch the
    next ones mid-tile (the masked case runs the K loop in 8 segments)."""
    p = Problem(dtype="fp8", seed=77, **case)
    g = p.gpu()
    out = bf16_to_f64(g.forward())
    assert g.status() == 0
    assert rel_fro(out, p.oracle_forward()) <= 2e-3
