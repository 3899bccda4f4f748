"""Tree-size choice (medusa_tree_size_choose): the size with the most expected tokens per
unit of step time, (1 + E[L](n)) / t(n), ties to the smaller size."""
import pytest

from medusa_head_speculative_gb300 import binding as Bnd

from harness import ensure_built


def test_picks_the_best_rate():
    ensure_built()
    e = [0.0, 0.7, 1.2, 1.5, 1.7]
    # rates 1.7, 2.0, 1.8 tokens/ms
    assert Bnd.tree_size_choose(e, [1, 2, 4], [1.0, 1.1, 1.5]) == 1
    # equal step times: the longer expected length wins
    assert Bnd.tree_size_choose(e, [2, 4, 1], [1.0, 1.0, 1.0]) == 1


def test_ties_go_to_the_smaller_tree():
    ensure_built()
    e = [0.0, 1.0, 3.0]
    assert Bnd.tree_size_choose(e, [1, 2], [1.0, 2.0]) == 0     # 2/1 == 4/2
    assert Bnd.tree_size_choose(e, [2, 1], [2.0, 1.0]) == 1


def test_cost_growing_with_size_moves_the_choice_down():
    """E[L](n) = 1 - q^n (one geometric head) with t(n) = 1 + c n: a larger c (a longer
    context makes every candidate dearer) never picks a larger tree."""
    ensure_built()
    q = 0.6
    e = [1 - q ** n for n in range(65)]
    sizes = [4, 8, 16, 32, 64]
    picks = [sizes[Bnd.tree_size_choose(e, sizes, [1 + c * n for n in sizes])]
             for c in (0.0, 0.002, 0.01, 0.05, 0.2)]
    assert picks[0] == 64 and picks == sorted(picks, reverse=True) and picks[-1] == 4


def test_rejects_bad_arguments():
    ensure_built()
    with pytest.raises(Bnd.MedusaError):
        Bnd.tree_size_choose([0.0, 1.0], [1], [0.0])
    with pytest.raises(Bnd.MedusaError):
        Bnd.tree_size_choose([0.0, 1.0], [2], [1.0])
