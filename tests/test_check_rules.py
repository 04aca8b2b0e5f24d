"""CPU tests of the comparison rules, with planted mistakes."""
import numpy as np
import pytest

from tests.msa_check import check_structure, compare_selection


def _case():
    # one row at position 5 * 8 + 3 (Bk = 8, loc = 5), k = 4, scores for blocks 0..5
    pos = np.array([43])
    ref = np.array([[[0, 2, 4, 5]]], dtype=np.int32)
    S = np.array([[[10.0, 1.0, 9.0, 2.0, 9.999, 0.0]]])
    return pos, ref, S


def test_exact_and_near_tie_swap_pass():
    pos, ref, S = _case()
    assert compare_selection(ref, ref, S, pos, 8) == 0
    S2 = S.copy()
    S2[0, 0, 3] = 9.995  # block 3 within 1e-3 of block 4 (9.999)
    gpu = np.array([[[0, 2, 3, 5]]], dtype=np.int32)
    assert compare_selection(gpu, ref, S2, pos, 8) == 1


@pytest.mark.parametrize("gpu", [
    [[[0, 2, 3, 5]]],   # swap with a large score gap
    [[[0, 2, 4, -1]]],  # local block missing
    [[[0, 2, 2, 5]]],   # duplicate
    [[[2, 0, 4, 5]]],   # not ascending
    [[[0, 2, 4, 6]]],   # block after the local one
    [[[0, 4, 5, -1]]],  # too few blocks
])
def test_planted_mistakes_fail(gpu):
    pos, ref, S = _case()
    with pytest.raises(AssertionError):
        compare_selection(np.array(gpu, dtype=np.int32), ref, S, pos, 8)


def test_structure_short_rows():
    check_structure(np.array([[[0, -1, -1]], [[0, 1, -1]]]), np.array([3, 9]), 8)
    with pytest.raises(AssertionError):
        check_structure(np.array([[[0, 1, -1]]]), np.array([3]), 8)
