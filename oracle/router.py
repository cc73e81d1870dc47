"""fp32 router: logits, top-k with a deterministic tie-break, and the
renormalised top-k weights (oracle; test use only).

"[Feature] Support BF16 and batch-invariant inference with DeepEP v2" (sglang
PR #38160 report), section "关联脉络": a companion change keeps the MoE router
GEMM in fp32 so that expert selection does not flip under deterministic
inference.  The layer consumes top-k expert ids and weights ("Support
DeepGEMM for standard MoE dispatch" (sglang PR #33128 report), "关键源码片段"
deep_gemm.py: standard top-k dispatch).  Readings adopted where the pages are
silent:

* logits z[t, e] = sum_k x[t, k] * W[e, k], x in bf16, W in fp32;
* the top-k experts by logit, descending, equal logits ordered by the lower
  expert id;
* weights = softmax over the selected logits (equivalently the full softmax
  renormalised over the top k).

Where a floating-point comparison decides an id, the oracle takes the
decision on the logits it is handed: ``select_topk`` is applied to the
kernel's own fp32 logits in the parity tests, while ``logits`` gives the fp64
reference values those logits are checked against.
"""

import numpy as np


def logits(x, w_router):
    """x [T, K] (bf16 values), w_router [E, K] (fp32 values) -> fp64 [T, E]."""
    return np.asarray(x, dtype=np.float64) @ np.asarray(w_router, dtype=np.float64).T


def select_topk(z, topk):
    """Top-k expert ids of each row of z, descending logit, ties to the lower
    id: a plain selection loop (k passes over the row)."""
    z = np.asarray(z)
    T, E = z.shape
    ids = np.zeros((T, topk), dtype=np.int64)
    for t in range(T):
        taken = np.zeros(E, dtype=bool)
        for j in range(topk):
            best = -1
            for e in range(E):
                if taken[e]:
                    continue
                if best < 0 or z[t, e] > z[t, best]:
                    best = e
            ids[t, j] = best
            taken[best] = True
    return ids


def topk_softmax(z, ids):
    """Softmax over the selected logits of each row, in fp64."""
    sel = np.take_along_axis(np.asarray(z, dtype=np.float64), ids, axis=1)
    ex = np.exp(sel - sel.max(axis=1, keepdims=True))
    return ex / ex.sum(axis=1, keepdims=True)


def route(x, w_router, topk):
    """The whole router in fp64: (ids [T, k], weights [T, k], logits [T, E])."""
    z = logits(x, w_router)
    ids = select_topk(z, topk)
    return ids, topk_softmax(z, ids), z
