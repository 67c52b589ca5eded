"""The literal-bar audit used by the GPU parity tests, checked on hand-made
BF16 bit patterns (no GPU needed)."""
import numpy as np

from tests import gpu_support as G


def _bits(*xs):
    return np.array(xs, dtype=np.uint16)


def test_one_step_above_two_is_counted_and_adjacent():
    # 2.0 = 0x4000; its upper neighbour 2.015625 = 0x4001 (difference 0.0156 > 1e-2)
    n, ok = G.literal_bar_audit(_bits(0x4001), _bits(0x4000))
    assert (n, ok) == (1, True)
    n, ok = G.literal_bar_audit(_bits(0xC001), _bits(0xC000))          # the same below -2
    assert (n, ok) == (1, True)


def test_two_steps_across_a_binade_are_not_adjacent():
    # 1.984375 = 0x3FFE is two steps below 2.0 (difference 0.0156, one step of 2.0)
    n, ok = G.literal_bar_audit(_bits(0x3FFE), _bits(0x4000))
    assert (n, ok) == (1, False)


def test_small_differences_are_not_counted():
    # 1.0 = 0x3F80 and its neighbour 1.0078125 = 0x3F81 differ by less than 1e-2
    n, ok = G.literal_bar_audit(_bits(0x3F81, 0x3F80), _bits(0x3F80, 0x3F80))
    assert (n, ok) == (0, True)


def test_opposite_signs_are_not_adjacent():
    # +2.0 vs -2.0 differ by 4
    n, ok = G.literal_bar_audit(_bits(0xC000), _bits(0x4000))
    assert (n, ok) == (1, False)
