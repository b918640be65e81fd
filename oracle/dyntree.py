"""Oracle of the EAGLE-2 dynamic draft tree: TEST INFRASTRUCTURE ONLY (tests, smoke and
the CPU leg of the benchmark may use it; the CUDA library never does).

EAGLE / EAGLE-2 paper translation (modelers.csdn.net), sections 2.3.1 and 2.3.2, and
"LLM speculative decoding: EAGLE" (jingming.pro), section 4.2.1:
  - the value of a draft token is the product of the draft model's confidences on the
    path from the root to it (its estimated global acceptance rate);
  - expansion: the draft model is fed the top-k tokens of the newest layer by value;
  - reranking: over all draft tokens, the top-m by value are kept, a shallower token
    winning a tie in value, so the kept tokens still form a connected tree;
  - the kept tokens are flattened to one sequence after the root, and the attention
    mask lets each token see only its ancestors (and itself).

Readings taken here (the pages leave them open):
  - values are fp32 products taken from the root down, v = v(parent) * p, rounded at
    every step (v(root) = 1);
  - candidates are numbered in creation order (layer by layer, within a layer by the
    order of the expanded parents, then by the child's rank); ties in value and depth
    go to the lower candidate number, which makes the selection unique;
  - the flattened order is breadth-first: by depth, then by candidate number (so
    siblings appear in the order the draft model ranked them), and a node's parent is
    its parent's position in that sequence; position id = depth.
"""
import numpy as np


def values_and_depths(cand_parent, cand_prob):
    """fp32 value and depth (root = 0) of every candidate; cand_parent[i] < i or -1."""
    n = len(cand_parent)
    val = np.zeros(n, dtype=np.float32)
    dep = np.zeros(n, dtype=np.int32)
    for i in range(n):
        p = int(cand_parent[i])
        pv = np.float32(1.0) if p < 0 else val[p]
        val[i] = np.float32(pv * np.float32(cand_prob[i]))
        dep[i] = 1 if p < 0 else dep[p] + 1
    return val, dep


def expand_topk(values, k):
    """Indices of the k largest values, ties to the lower index (the expansion step)."""
    order = sorted(range(len(values)), key=lambda i: (-float(values[i]), i))
    return order[:k]


def build_tree(cand_parent, cand_token, cand_prob, root_token, m):
    """Select m draft tokens and flatten them.  Returns dict with tokens, parent_idx,
    position_ids, src (candidate of each position, -1 for the root) of length m + 1
    and the (m + 1) x (m + 1) ancestor mask (uint8)."""
    val, dep = values_and_depths(cand_parent, cand_prob)
    n = len(cand_parent)
    ranked = sorted(range(n), key=lambda i: (-float(val[i]), int(dep[i]), i))
    keep = set(ranked[:m])
    flat = sorted(keep, key=lambda i: (int(dep[i]), i))
    pos = {c: j + 1 for j, c in enumerate(flat)}
    M = m + 1
    tokens = np.zeros(M, dtype=np.int32)
    parent = np.full(M, -1, dtype=np.int32)
    depth = np.zeros(M, dtype=np.int32)
    src = np.full(M, -1, dtype=np.int32)
    tokens[0] = root_token
    for j, c in enumerate(flat, start=1):
        tokens[j] = cand_token[c]
        p = int(cand_parent[c])
        parent[j] = 0 if p < 0 else pos[p]
        depth[j] = dep[c]
        src[j] = c
    mask = np.zeros((M, M), dtype=np.uint8)
    for j in range(M):
        a = j
        while a >= 0:
            mask[j, a] = 1
            a = parent[a]
    return {"tokens": tokens, "parent_idx": parent, "position_ids": depth, "src": src,
            "mask": mask}
