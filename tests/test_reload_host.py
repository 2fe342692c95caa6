"""The time model of the double-buffered reload (no GPU): the pages' closed
form c + (L-1) max(c, g) + g for alike layers, L (c + g) for one buffer."""
import pytest

from qlora_fine_tuning_gb300.reload import model_double_buffer, model_single_buffer


@pytest.mark.parametrize("c,g,L", [(1.0, 2.0, 3), (2.0, 1.0, 5), (1.5, 1.5, 1), (0.3, 0.7, 28)])
def test_alike_layers_follow_the_closed_form(c, g, L):
    assert model_double_buffer([c] * L, [g] * L) == pytest.approx(c + (L - 1) * max(c, g) + g)
    assert model_single_buffer([c] * L, [g] * L) == pytest.approx(L * (c + g))
    # what the second buffer saves: (L-1) min(c, g)
    saved = model_single_buffer([c] * L, [g] * L) - model_double_buffer([c] * L, [g] * L)
    assert saved == pytest.approx((L - 1) * min(c, g))


def test_unequal_layers_overlap_each_copy_with_the_previous_compute():
    # copy of layer k overlaps compute of layer k-1
    assert model_double_buffer([1.0, 4.0, 1.0], [2.0, 1.0, 3.0]) == pytest.approx(1.0 + 4.0 + 1.0 + 3.0)
    assert model_double_buffer([], []) == 0.0
