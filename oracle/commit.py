"""Oracle of the accepted-path commit: TEST INFRASTRUCTURE ONLY (tests, smoke and the
CPU leg of the benchmark may use it; the CUDA library never does).

After a verify step the cache entries of the whole draft tree sit after each
sequence's prefix, node n of tree b at position prefix_len[b] + n; the entries of
the accepted path are kept and moved to consecutive positions, so that the caches
continue the accepted sequence ("EAGLE close reading", edgeai1.github.io, section 5:
after a rejection both caches are trimmed to what was accepted -- the cache
rearrangement step of a decoding round).

Reading taken here (the page names the step, not its layout): position
prefix_len[b] + k receives node path[b][k] for k = 0 .. accept_len[b], one move after
the other in increasing k; every other position keeps its bytes; a tree with
accept_len < 0 (a failed tree) is left as it is.
"""
import numpy as np


def commit_accepted_path(cache: np.ndarray, prefix_len, accepted_path, accept_len):
    """cache [planes, B, positions, row_bytes] (uint8); returns the committed copy."""
    out = np.array(cache, copy=True)
    P, B, n_pos, _ = out.shape
    for b in range(B):
        a = int(accept_len[b])
        if a < 0:
            continue
        base = int(prefix_len[b])
        for k in range(1, a + 1):
            src = base + int(accepted_path[b][k])
            dst = base + k
            if src < n_pos and dst < n_pos:
                out[:, b, dst, :] = out[:, b, src, :]
    return out
