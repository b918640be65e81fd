"""The accepted-path commit oracle against hand-worked results (the definition: position
prefix + k receives node path[k], one move after the other)."""
import numpy as np

from oracle.commit import commit_accepted_path


def _cache(P, B, n_pos, row):
    # every row holds its own (plane, tree, position) label in its first three bytes
    c = np.zeros((P, B, n_pos, row), dtype=np.uint8)
    for p in range(P):
        for b in range(B):
            for t in range(n_pos):
                c[p, b, t, :3] = (p, b, t)
    return c


def test_overlapping_moves_take_sources_before_they_are_overwritten():
    c = _cache(1, 1, 12, 16)
    out = commit_accepted_path(c, [5], [[0, 2, 3, -1]], [2])
    # position 6 <- node 2 (old position 7), position 7 <- node 3 (old position 8)
    assert out[0, 0, 6, 2] == 7 and out[0, 0, 7, 2] == 8
    keep = [t for t in range(12) if t not in (6, 7)]
    np.testing.assert_array_equal(out[0, 0, keep], c[0, 0, keep])


def test_contiguous_path_is_a_no_op_and_failed_or_empty_trees_are_untouched():
    c = _cache(2, 3, 10, 32)
    out = commit_accepted_path(c, [1, 2, 3], [[0, 1, 2], [0, 4, -1], [0, 3, 5]], [2, 0, -1])
    np.testing.assert_array_equal(out, c)


def test_planes_and_trees_move_independently():
    c = _cache(3, 2, 16, 16)
    out = commit_accepted_path(c, [4, 0], [[0, 3, 9, 11], [0, 5, -1, -1]], [3, 1])
    for p in range(3):
        assert [out[p, 0, t, 2] for t in (5, 6, 7)] == [7, 13, 15]
        assert out[p, 1, 1, 2] == 5
        assert out[p, 0, 4, 2] == 4 and out[p, 1, 0, 2] == 0  # roots stay
        assert out[p, 1, 2, 2] == 2                           # beyond the path: unchanged


def test_moves_beyond_the_cache_are_skipped():
    c = _cache(1, 1, 8, 16)
    out = commit_accepted_path(c, [6], [[0, 1, 3]], [2])
    assert out[0, 0, 7, 2] == 7  # 7 <- 7: in place; 8 <- 9 lies beyond: skipped
    np.testing.assert_array_equal(out[0, 0, :7], c[0, 0, :7])
