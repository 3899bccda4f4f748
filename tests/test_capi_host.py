"""Host-side checks of the C ABI that need no GPU: the library loads and exports every
declared entry point, the host tree builders agree exactly with the oracle's, and plan
validation rejects malformed inputs before any CUDA call."""
import os
import re

import numpy as np
import pytest

import oracle as O
import synthetic as S
from medusa_head_speculative_gb300 import binding as Bnd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(Bnd.LIB_PATH):
        from medusa_head_speculative_gb300 import build
        build.build()
    return Bnd.lib()


def declared_functions():
    names = []
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if not f.endswith(".h"):
            continue
        text = open(os.path.join(inc, f)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:[\w\s\*]+?)\b(medusa_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_library_exports_every_declared_symbol(L):
    names = declared_functions()
    assert len(names) >= 15
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing


@pytest.mark.parametrize("s", [(3, 2, 2), (2, 3), (1,), (4, 1, 3, 2), (8, 8)])
def test_cartesian_builder_matches_oracle(L, s):
    parent, rank = Bnd.tree_cartesian(s)
    spec = O.cartesian_tree(s)
    assert list(parent) == spec.parent and list(rank) == spec.rank


@pytest.mark.parametrize("K,N", [(5, 64), (4, 42), (5, 16), (5, 128), (3, 7)])
def test_greedy_builder_matches_oracle(L, K, N):
    a = S.score_table(K, 10)
    parent, rank = Bnd.tree_greedy((10,) * K, a, N)
    spec = O.greedy_tree(a, (10,) * K, N)
    assert list(parent) == spec.parent and list(rank) == spec.rank


@pytest.mark.parametrize("seed", range(6))
def test_greedy_builder_matches_oracle_random_tables(L, seed):
    rng = np.random.default_rng(seed)
    K, smax = 4, 5
    a = np.round(rng.random((K, smax)), 1)        # coarse values: many exact ties
    s = tuple(int(x) for x in rng.integers(1, smax + 1, size=K))
    N = int(rng.integers(1, 30))
    parent, rank = Bnd.tree_greedy(s, a, N)
    spec = O.greedy_tree(a, s, N)
    assert list(parent) == spec.parent and list(rank) == spec.rank


def _plan(**kw):
    args = dict(B=1, d=128, V=512, K=3, Hq=4, Hkv=4, dh=32, dtype=Bnd.F32, capacity=128,
                s=(3, 2, 2))
    parent, rank = Bnd.tree_cartesian(args["s"])
    args.update(parent=parent, rank=rank)
    args.update(kw)
    return Bnd.Plan(**args)


@pytest.mark.parametrize("bad,code", [
    (dict(Hkv=3), Bnd.MEDUSA_ERR_INVALID),                        # Hq % Hkv != 0
    (dict(dh=48), Bnd.MEDUSA_ERR_UNSUPPORTED),
    (dict(d=130), Bnd.MEDUSA_ERR_UNSUPPORTED),                     # not a 16-byte multiple
    (dict(parent=np.array([-1, 0, 2, 1], np.int32), rank=np.array([0, 0, 0, 0], np.int32)),
     Bnd.MEDUSA_ERR_INVALID),                                      # parent >= own index
    (dict(parent=np.array([-1, 0, 1, 2, 3], np.int32), rank=np.array([0, 0, 0, 0, 0], np.int32)),
     Bnd.MEDUSA_ERR_INVALID),                                      # depth > K
    (dict(parent=np.array([-1, 0], np.int32), rank=np.array([0, 3], np.int32)),
     Bnd.MEDUSA_ERR_INVALID),                                      # rank >= s_1
    (dict(parent=np.array([-1, 0, 0], np.int32), rank=np.array([0, 1, 1], np.int32)),
     Bnd.MEDUSA_ERR_INVALID),                                      # duplicate child
    (dict(K=9, s=(1,) * 9, parent=np.array([-1], np.int32), rank=np.array([0], np.int32)),
     Bnd.MEDUSA_ERR_UNSUPPORTED),
    (dict(page_size=16, capacity=100, num_pages=8), Bnd.MEDUSA_ERR_INVALID),
    (dict(dtype=7), Bnd.MEDUSA_ERR_INVALID),
])
def test_plan_validation_rejects_before_any_cuda_call(L, bad, code):
    with pytest.raises(Bnd.MedusaError) as e:
        _plan(**bad)
    assert e.value.code == code


def test_too_many_nodes_unsupported(L):
    parent = np.concatenate([[-1], np.zeros(256, np.int32)]).astype(np.int32)
    rank = np.concatenate([[0], np.arange(256) % 16]).astype(np.int32)
    with pytest.raises(Bnd.MedusaError) as e:
        _plan(K=1, s=(16,), parent=parent, rank=rank)
    assert e.value.code == Bnd.MEDUSA_ERR_UNSUPPORTED
