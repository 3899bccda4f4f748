"""The optimized tree built on the device (medusa_tree_greedy_device) equals the oracle's
greedy construction and the host builder index for index, and its expected-length curve
equals the oracle's E[L] of the nested greedy trees and, for one head with geometric
accuracies, the closed form 1 - (1 - t)^n."""
import numpy as np
import pytest
import torch

import oracle as O
import synthetic as S
from medusa_head_speculative_gb300 import binding as Bnd

from harness import ensure_built

pytestmark = pytest.mark.gpu


def _device_tree(s, a, N):
    a_dev = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64)).cuda()
    parent = torch.full((N + 1,), -9, dtype=torch.int32, device="cuda")
    rank = torch.full((N + 1,), -9, dtype=torch.int32, device="cuda")
    exp = torch.full((N + 1,), -1.0, dtype=torch.float64, device="cuda")
    Bnd.tree_greedy_device(list(s), a_dev, N, parent, rank, exp)
    torch.cuda.synchronize()
    return parent.cpu().numpy(), rank.cpu().numpy(), exp.cpu().numpy()


def _tables():
    rng = np.random.default_rng(5)
    out = [("geometric_5x10", (10,) * 5, S.score_table(5, 10), [1, 16, 64, 128, 255])]
    a = rng.random((4, 8))                                   # not monotone in rank
    out.append(("random_4x8", (8, 6, 8, 5), a, [1, 37, 100, 200]))
    ties = rng.choice([0.5, 0.25, 0.125, 1.0], size=(3, 6))  # many equal path products
    out.append(("ties_3x6", (6, 6, 6), ties, [5, 50, 150, 258 - 36]))
    out.append(("cartesian_full", (3, 2), np.array([[0.6, 0.3, 0.1], [0.5, 0.5, 0.0]]), [9]))
    big = rng.random((8, 16)) * 0.9 + 0.05
    out.append(("max_8x16", (16,) * 8, big, [255]))
    return out


@pytest.mark.parametrize("name,s,a,Ns", _tables(), ids=[t[0] for t in _tables()])
def test_device_tree_equals_oracle_and_host(name, s, a, Ns):
    ensure_built()
    for N in Ns:
        parent, rank, exp = _device_tree(s, a, N)
        spec = O.greedy_tree(a, list(s), N)
        assert spec.N == N
        assert list(parent) == list(spec.parent), (name, N)
        assert list(rank) == list(spec.rank), (name, N)
        hp, hr = Bnd.tree_greedy(list(s), a, N)
        assert list(parent) == list(hp) and list(rank) == list(hr)
        # the curve: expected[n] = E[L] of the greedy tree of n nodes (trees are nested)
        for n in sorted({0, 1, N // 3, N // 2, N}):
            ref = 0.0 if n == 0 else O.expected_accept_length(O.greedy_tree(a, list(s), n), a)
            assert abs(exp[n] - ref) <= 1e-12 * max(1.0, ref), (name, N, n)


def test_expected_length_closed_form_one_head():
    """One head whose rank-i accuracy is t (1 - t)^i: the greedy tree takes ranks 0..n-1 and
    E[L](n) = sum_i t (1 - t)^i = 1 - (1 - t)^n."""
    ensure_built()
    t, N = 0.37, 16
    a = np.array([[t * (1 - t) ** i for i in range(N)]])
    parent, rank, exp = _device_tree((N,), a, N)
    assert list(parent) == [-1] + [0] * N and list(rank) == [0] + list(range(N))
    for n in range(N + 1):
        assert abs(exp[n] - (1 - (1 - t) ** n)) <= 1e-12


def test_device_tree_rejects_bad_sizes():
    ensure_built()
    a = torch.zeros(2, 3, dtype=torch.float64, device="cuda")
    p = torch.empty(20, dtype=torch.int32, device="cuda")
    with pytest.raises(Bnd.MedusaError):
        Bnd.tree_greedy_device([3, 2], a, 10, p, p)          # the Cartesian tree has 9 nodes
    with pytest.raises(Bnd.MedusaError):
        Bnd.tree_greedy_device([3, 4], a, 5, p, p)           # s[1] > smax
