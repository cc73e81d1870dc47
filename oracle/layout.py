"""Per-expert row layouts (oracle; test use only).

Sources: "Support DeepGEMM for standard MoE dispatch" (sglang PR #33128
report), sections "实现拆解" steps 2-4 and "关键源码片段" (deep_gemm.py,
ep_moe_kernels.py); "[Feature] Support BF16 and batch-invariant inference
with DeepEP v2" (sglang PR #38160 report), "实现拆解" step 1 (local expert
range given by ``expert_start`` and the local expert count).

Readings adopted where the reports are silent:

* ``m_indices`` holds the *local* expert index (the scatter kernel shown in
  the report writes its own program id, one program per local expert).
* Rows after the last expert segment, up to the static bound, are ``-1`` too,
  so every row that carries no token is ``-1``.
* Inside an expert segment, assignments are ordered by their flattened
  position ``t * topk + j`` (a stable counting sort); the reports do not fix
  the order, and this one is deterministic.
* Ids of ``-1`` and ids outside ``[expert_start, expert_start + E_local)``
  are dropped (``src2dst = -1``).  Ids below -1 or >= E_global are data
  errors: they are dropped and reported.
* Masked layout: expert e's assignments occupy rows ``e * max_m + rank``;
  ``masked_m[e]`` is the number of them.  An expert with more than ``max_m``
  assignments overflows: the extra ones are dropped and reported.
"""

import numpy as np


def use_masked_layout(num_experts, num_local_experts):
    """Layout choice of the standard-dispatch runner ("关键源码片段"
    deep_gemm.py): masked when experts are sharded (more experts than local
    ones) and at most 32 are local, compact otherwise."""
    return num_experts > num_local_experts and num_local_experts <= 32


def compact_all_tokens(num_assignments, num_experts, block_e=128):
    """Static row count of the compact layout ("关键源码片段" deep_gemm.py):
    every non-empty expert takes at least one block of ``block_e`` rows, and
    the assignments beyond one per non-empty expert fill whole extra blocks.
    The worst case has min(A, E) non-empty experts."""
    nonempty = min(num_assignments, num_experts)
    return block_e * (nonempty + (num_assignments - nonempty) // block_e)


def plan_layout(topk_ids, E_global, E_local, expert_start, layout, block_e=128, max_m=None):
    """Compute the dispatch layout for ``topk_ids`` [T, topk].

    layout: "compact" or "masked".  Returns a dict with
      counts   [E_local]          assignments per local expert
      src2dst  [T, topk]          destination row of each assignment, -1 if dropped
      errors   set of str         {"expert_id", "masked_overflow"} data errors seen
    and, for "compact":
      padded   [E_local]          counts rounded up to a multiple of block_e
      start    [E_local]          exclusive prefix sum of padded
      all_tokens                  static row bound (compact_all_tokens)
      m_indices [all_tokens]      local expert of each row, -1 on rows without a token
    or, for "masked":
      masked_m [E_local]          valid rows of each expert (== counts unless overflow)
    """
    ids = np.asarray(topk_ids, dtype=np.int64)
    T, k = ids.shape
    flat = ids.reshape(-1)
    errors = set()

    # 1. local expert of every assignment (or -1 when dropped)
    local = np.full(flat.shape, -1, dtype=np.int64)
    for i, gid in enumerate(flat):
        if gid < -1 or gid >= E_global:
            errors.add("expert_id")
            continue
        if gid == -1:
            continue
        e = gid - expert_start
        if 0 <= e < E_local:
            local[i] = e

    # 2. stable rank of every assignment inside its expert (flattened order)
    counts = np.zeros(E_local, dtype=np.int64)
    rank = np.full(flat.shape, -1, dtype=np.int64)
    for i, e in enumerate(local):
        if e >= 0:
            rank[i] = counts[e]
            counts[e] += 1

    out = {"counts": counts, "errors": errors}
    src2dst = np.full(flat.shape, -1, dtype=np.int64)

    if layout == "compact":
        padded = (counts + block_e - 1) // block_e * block_e
        start = np.concatenate([[0], np.cumsum(padded)[:-1]]).astype(np.int64)
        all_tokens = compact_all_tokens(int(local.size), E_local, block_e)
        m_indices = np.full(all_tokens, -1, dtype=np.int64)
        for e in range(E_local):
            # the first counts[e] rows of the segment carry tokens, the rest are padding
            m_indices[start[e]:start[e] + counts[e]] = e
        for i, e in enumerate(local):
            if e >= 0:
                src2dst[i] = start[e] + rank[i]
        out.update(padded=padded, start=start, all_tokens=all_tokens, m_indices=m_indices)
    elif layout == "masked":
        if max_m is None:
            raise ValueError("masked layout needs max_m")
        masked_m = np.minimum(counts, max_m)
        if np.any(counts > max_m):
            errors.add("masked_overflow")
        for i, e in enumerate(local):
            if e >= 0 and rank[i] < max_m:
                src2dst[i] = e * max_m + rank[i]
        out.update(masked_m=masked_m, max_m=max_m)
    else:
        raise ValueError(f"unknown layout {layout!r}")

    out["src2dst"] = src2dst.reshape(T, k)
    return out
