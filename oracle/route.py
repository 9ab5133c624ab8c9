"""Token-to-expert grouping (oracle; test infrastructure only).

``Mxfp4MoEMethod.apply`` (vLLM quantization/mxfp4 API page) hands the fused-MoE
kernel ``topk_ids`` and ``topk_weights`` of shape [T, topk]; the kernel groups
the T*topk (token, slot) pairs by expert before the two grouped GEMMs.  The
pages give no algorithm for this step; the reading used here is a stable
counting sort of the flat pair index p = t*topk + k by expert id.  Ids outside
[0, E) (the ``expert_map`` -1 convention for non-local experts) join no group.
Duplicate ids in one row are separate pairs.

Expert parallelism (``apply`` passes ``global_num_experts`` and
``expert_map``): with a map, the ids in ``topk_ids`` are global expert ids in
[0, global_num_experts); ``expert_map[g]`` is the local id of global expert g
on this GPU, or -1 when another GPU holds it.  The pages print no formula for
the lookup; the plain reading is used: a global id outside the map, or one the
map sends to -1, joins no group, exactly like an invalid local id.
"""

from __future__ import annotations

import numpy as np


def local_ids(topk_ids: np.ndarray, expert_map=None) -> np.ndarray:
    """Global expert ids -> local ids through ``expert_map`` (int64 array; -1
    for non-local or out-of-range ids).  Without a map the ids are returned as
    they are (already local)."""
    ids = np.asarray(topk_ids).astype(np.int64)
    if expert_map is None:
        return ids
    emap = np.asarray(expert_map).astype(np.int64)
    inside = (ids >= 0) & (ids < emap.size)
    out = np.full(ids.shape, -1, dtype=np.int64)
    out[inside] = emap[ids[inside]]
    return out


def route(topk_ids: np.ndarray, E: int, expert_map=None):
    """Group pairs by expert.

    Returns ``(counts int32[E], offsets int32[E+1], sorted_pair int32[P],
    pair_pos int32[P])``: ``sorted_pair[offsets[e]:offsets[e+1]]`` lists expert
    e's pairs in ascending flat index; entries past ``offsets[E]`` are -1.
    ``pair_pos[p]`` is the position of pair p in ``sorted_pair`` (-1 if invalid).
    """
    ids = local_ids(topk_ids, expert_map).reshape(-1)
    P = ids.size
    valid = (ids >= 0) & (ids < E)
    counts = np.bincount(ids[valid], minlength=E).astype(np.int32)
    offsets = np.zeros(E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    n_valid = int(offsets[-1])
    key = np.where(valid, ids, E)
    order = np.argsort(key, kind="stable")
    sorted_pair = np.full(P, -1, dtype=np.int32)
    sorted_pair[:n_valid] = order[:n_valid]
    pair_pos = np.full(P, -1, dtype=np.int32)
    pair_pos[order[:n_valid]] = np.arange(n_valid, dtype=np.int32)
    return counts, offsets, sorted_pair, pair_pos


def router_topk(logits: np.ndarray, topk: int, renormalize: bool = True):
    """Top-k routing from router logits, float64.

    The Mxfp4MoEMethod page's ``apply_monolithic`` hands the kernel
    ``router_logits`` and lets it choose each token's experts; the pages print
    no scoring formula.  The plain reading used here (the one that turns the
    logits into the top-k ids and weights ``apply`` takes): p = softmax over
    the experts of each token's logits; keep the ``topk`` largest p, ties to
    the lower expert id; with ``renormalize`` the kept p are divided by their
    sum.  Grouped top-k, a score-correction bias and a routed scaling factor
    are not modelled.

    Returns ``ids int32[T, topk]`` (in decreasing p) and ``w float32[T, topk]``
    (the float64 result rounded to float32 once).
    """
    L = np.asarray(logits, dtype=np.float64)
    T, G = L.shape
    ids = np.zeros((T, topk), dtype=np.int32)
    w = np.zeros((T, topk), dtype=np.float64)
    for t in range(T):
        e = np.exp(L[t] - L[t].max())
        p = e / e.sum()
        # decreasing p; among equal p the lower id first
        order = sorted(range(G), key=lambda i: (-p[i], i))[:topk]
        ids[t] = order
        w[t] = p[order] / p[order].sum() if renormalize else p[order]
    return ids, w.astype(np.float32)


def active_experts(counts: np.ndarray) -> np.ndarray:
    """Ids of experts that received at least one pair, ascending."""
    return np.nonzero(np.asarray(counts) > 0)[0].astype(np.int32)
