"""Oracle of the draft-side top-k drafting step: TEST INFRASTRUCTURE ONLY (tests, smoke
and the CPU leg of the benchmark may use it; the CUDA library never does).

EAGLE / EAGLE-2 paper translation (modelers.csdn.net), sections 2.3.1-2.3.2, and "LLM
speculative decoding: EAGLE" (jingming.pro), section 4.2.1: the draft model's
distribution at a node proposes its top-k tokens as that node's children, each with
the draft model's confidence (its probability), which the dynamic tree multiplies
along a path.

Readings taken here (the pages leave them open):
  - the k children are the k largest draft logits, ties to the lower vocabulary index,
    listed in that order (the rank order the dynamic tree keeps for siblings);
  - a child's confidence is its softmax probability at temperature T over the whole
    row, exp((z - max)/T) / sum over the row of exp((z' - max)/T), in fp64;
  - a row holding NaN or +inf, or all -inf, has no draft: status 1, tokens -1,
    confidences 0.
"""
import numpy as np


def _as_f64(row):
    row = np.asarray(row)
    if row.dtype == np.uint16:  # raw bf16 bits
        return (row.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return row.astype(np.float32).astype(np.float64)


def draft_topk(logits, k: int, temperature: float):
    """logits [R, V] (float32, or uint16 raw bf16 bits).  Returns tokens [R, k] int32,
    probs [R, k] float64 and status [R] int32."""
    logits = np.atleast_2d(np.asarray(logits))
    R = logits.shape[0]
    tokens = np.full((R, k), -1, dtype=np.int32)
    probs = np.zeros((R, k), dtype=np.float64)
    status = np.zeros(R, dtype=np.int32)
    for r in range(R):
        z = _as_f64(logits[r])
        m = z.max() if z.size else -np.inf
        if np.isnan(z).any() or m == np.inf or m == -np.inf:
            status[r] = 1
            continue
        order = sorted(range(len(z)), key=lambda i: (-z[i], i))[:k]
        w = np.exp((z - m) / temperature)
        s = w.sum()
        tokens[r, :len(order)] = order
        probs[r, :len(order)] = w[order] / s
    return tokens, probs, status
