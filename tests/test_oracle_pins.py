"""Pins of the fp64 oracle to facts fixed by the pages and by mathematics.

None of these re-types the oracle's own formula: each checks a closed form, a special
case that reduces to a textbook or library routine, an invariant, a value printed on
the pages (tests/golden/) or a brute force on a tiny input.
"""
import itertools
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle as O
import synthetic as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    rows = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.split("#")[0].strip()
        if line:
            rows.append(line.split())
    return rows


# ------------------------------------------------------------------ heads
def test_silu_matches_library_sigmoid():
    x = np.linspace(-30, 30, 601)
    np.testing.assert_allclose(O.silu(x), x * scipy.special.expit(x), rtol=1e-14, atol=1e-300)
    assert O.silu(np.array([0.0]))[0] == 0.0


def test_head_at_initialisation_equals_lm_head():
    """W1 = 0 and W2 = LM head: SiLU(0) = 0, the residual passes h through, and the
    head's prediction equals the LM head's exactly (Medusa summary §3.4 'Why this form')."""
    rng = np.random.default_rng(1)
    d, V = 48, 97
    LM = rng.standard_normal((V, d))
    h = rng.standard_normal(d)
    u, z = O.medusa_head(np.zeros((d, d)), LM, h)
    np.testing.assert_array_equal(u, h)
    np.testing.assert_array_equal(z, O.lm_head(LM, h))


def test_head_brute_force_loops():
    """Orientation and residual: W2 [V][d] rows dotted with SiLU(W1 h) + h, by loops."""
    rng = np.random.default_rng(2)
    d, V = 6, 9
    W1, W2, h = rng.standard_normal((d, d)), rng.standard_normal((V, d)), rng.standard_normal(d)
    u_ref = [0.0] * d
    for i in range(d):
        a = sum(W1[i][j] * h[j] for j in range(d))
        u_ref[i] = a / (1 + math.exp(-a)) + h[i]
    z_ref = [sum(W2[v][j] * u_ref[j] for j in range(d)) for v in range(V)]
    u, z = O.medusa_head(W1, W2, h)
    np.testing.assert_allclose(u, u_ref, rtol=1e-13)
    np.testing.assert_allclose(z, z_ref, rtol=1e-12, atol=1e-13)


def test_head_param_count_golden():
    (d, V, per_head, five), = _golden_rows("head_params.txt")
    d, V = int(d), int(V)
    # the page adds its rounded parts (16.8M + 131.1M), so allow that rounding
    assert abs((d * d + d * V) / 1e6 - float(per_head)) <= 0.1
    assert abs(5 * (d * d + d * V) / 1e6 - float(five)) < 1.0


def test_topk_brute_force_with_ties():
    z = np.array([1.0, 3.0, 3.0, 2.0, 3.0, -1.0, 2.0])
    idx, val, mar = O.top_s(z, 4)
    assert list(idx) == [1, 2, 4, 3]          # equal values: lower index first
    assert list(val) == [3.0, 3.0, 3.0, 2.0]
    assert mar[0] == 0.0 and mar[3] == 0.0    # 2.0 ties with index 6
    rng = np.random.default_rng(3)
    for _ in range(20):
        z = rng.integers(0, 6, size=40).astype(float)     # many ties
        s = int(rng.integers(1, 10))
        idx, _, _ = O.top_s(z, s)
        ref = sorted(range(40), key=lambda v: (-z[v], v))[:s]
        assert list(idx) == ref
        # every kept value >= every dropped value
        assert z[idx].min() >= np.delete(z, idx).max()


def test_argmax_lowest_index_on_ties():
    z = np.array([0.5, 2.0, -1.0, 2.0, 2.0])
    best, margin = O.argmax_lowest(z)
    assert best == 1 and margin == 0.0
    best, margin = O.argmax_lowest(np.array([0.0, 1.0, 0.25]))
    assert best == 1 and margin == 0.75


# ------------------------------------------------------------------ tree
@pytest.mark.parametrize("row", _golden_rows("node_counts.txt"))
def test_cartesian_node_and_path_counts(row):
    s = [int(x) for x in row[0].split(",")]
    spec = O.cartesian_tree(s)
    assert spec.N == int(row[1])
    assert len(O.retrieve_paths(spec)) == int(row[2])
    # closed form sum_k prod_{i<=k} s_i, level k holds prod_{i<=k} s_i nodes
    assert spec.N == sum(math.prod(s[:k + 1]) for k in range(len(s)))
    for k in range(1, len(s) + 1):
        assert sum(1 for dd in spec.depth if dd == k) == math.prod(s[:k])


def _check_tree_invariants(spec, L=37):
    n1 = spec.N + 1
    M = O.tree_mask(spec)
    pos = O.tree_positions(spec, L)
    assert spec.parent[0] == -1 and spec.depth[0] == 0
    for i in range(1, n1):
        p = spec.parent[i]
        assert 0 <= p < i
        assert spec.depth[i] == spec.depth[p] + 1
        row = M[p].copy()
        row[i] = 1
        np.testing.assert_array_equal(M[i], row)          # mask[i] = mask[parent] + {i}
    assert np.all(np.triu(M, 1) == 0)                      # lower triangular
    assert np.all(np.diag(M) == 1)
    np.testing.assert_array_equal(M.sum(1), np.array(spec.depth) + 1)
    np.testing.assert_array_equal(pos - L, M.sum(1) - 1)  # position = t + depth
    # M[i][j] = 1 iff j lies on the path i -> root, by walking parents
    for i in range(n1):
        anc, j = set(), i
        while j >= 0:
            anc.add(j)
            j = spec.parent[j]
        for j in range(n1):
            assert M[i, j] == (1 if j in anc else 0)
    # retrieve paths: one per leaf, each a parent chain from the root
    leaves = [n for n in range(n1) if n not in set(spec.parent[1:])]
    paths = O.retrieve_paths(spec)
    assert [p[-1] for p in paths] == leaves
    for p in paths:
        assert p[0] == 0 and all(spec.parent[p[t + 1]] == p[t] for t in range(len(p) - 1))


@pytest.mark.parametrize("s", [(3, 2, 2), (2, 3), (1,), (4, 1, 3, 2)])
def test_cartesian_tree_invariants(s):
    _check_tree_invariants(O.cartesian_tree(s))


def _closed_subsets(K, smax, N):
    """All ancestor-closed sets of N rank paths (brute force)."""
    allp = [p for k in range(1, K + 1) for p in itertools.product(range(smax), repeat=k)]
    for combo in itertools.combinations(allp, N):
        c = set(combo)
        if all(p[:-1] in c or len(p) == 1 for p in c):
            yield c


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("N", [1, 3, 5, 6])
def test_greedy_tree_is_the_brute_force_optimum(seed, N):
    """Greedy by path product maximises E[L] = sum over nodes of prod a
    (Notes on Medusa, section 4) among all trees with N nodes."""
    rng = np.random.default_rng(seed)
    K, smax = 3, 3
    a = np.sort(rng.random((K, smax)) * 0.9, axis=1)[:, ::-1]
    spec = O.greedy_tree(a, [smax] * K, N)
    assert spec.N == N
    _check_tree_invariants(spec)
    best = max(O.expected_accept_length(O.pack_tree(c), a)
               for c in _closed_subsets(K, smax, N))
    assert abs(O.expected_accept_length(spec, a) - best) < 1e-12


def test_greedy_equals_cartesian_when_budget_covers_it():
    a = S.score_table(3, 3)
    full = O.cartesian_tree((3, 3, 3))
    g = O.greedy_tree(a, (3, 3, 3), full.N)
    assert g.paths == full.paths


@pytest.mark.parametrize("K,N,depth", [(5, 64, 5), (4, 42, 4), (5, 16, 4), (5, 128, 5)])
def test_workload_trees_reach_stated_depth(K, N, depth):
    spec = O.greedy_tree(S.score_table(K, 10), (10,) * K, N)
    assert spec.N == N and max(spec.depth) == depth
    _check_tree_invariants(spec)


# ------------------------------------------------------------------ layer pieces
def test_rope_closed_forms():
    rng = np.random.default_rng(5)
    x, y = rng.standard_normal(16), rng.standard_normal(16)
    np.testing.assert_allclose(O.rope(x, 0, 10000.0), x, rtol=0, atol=0)
    np.testing.assert_allclose(np.linalg.norm(O.rope(x, 123, 10000.0)), np.linalg.norm(x), rtol=1e-14)
    # relative-position property: <R_m x, R_n y> depends only on m - n
    a = O.rope(x, 40, 10000.0) @ O.rope(y, 33, 10000.0)
    b = O.rope(x, 1007, 10000.0) @ O.rope(y, 1000, 10000.0)
    assert abs(a - b) < 1e-10
    # first pair rotates by exactly pos radians (theta_0 = 1)
    e = np.zeros(16)
    e[0] = 1.0
    r = O.rope(e, 2, 10000.0)
    assert abs(r[0] - math.cos(2)) < 1e-15 and abs(r[8] - math.sin(2)) < 1e-15


def test_attend_closed_forms():
    rng = np.random.default_rng(6)
    vals = rng.standard_normal((5, 4))
    # one key: the output is its value
    np.testing.assert_allclose(O.attend(rng.standard_normal(4), rng.standard_normal((1, 4)), vals[:1]), vals[0])
    # equal scores: the mean of the values
    np.testing.assert_allclose(O.attend(np.zeros(4), rng.standard_normal((5, 4)), vals), vals.mean(0), rtol=1e-14)
    # against scipy's softmax
    q, keys = rng.standard_normal(4), rng.standard_normal((5, 4))
    ref = scipy.special.softmax(keys @ q / 2.0) @ vals
    np.testing.assert_allclose(O.attend(q, keys, vals), ref, rtol=1e-13)


@pytest.mark.parametrize("s,Hq,Hkv", [((3, 2, 2), 4, 4), ((2, 3), 4, 2), ((1,), 2, 1)])
def test_tree_attention_equals_per_path_causal_attention(s, Hq, Hkv):
    """Every node's output equals plain attention over prefix + its own root->node path,
    computed on its own (the tree mask's purpose, Medusa summary §3.4 Step 3)."""
    rng = np.random.default_rng(7)
    spec = O.cartesian_tree(s)
    n1, dh, L = spec.N + 1, 8, 11
    q = rng.standard_normal((n1, Hq, dh))
    kc, vc = rng.standard_normal((L, Hkv, dh)), rng.standard_normal((L, Hkv, dh))
    kt, vt = rng.standard_normal((n1, Hkv, dh)), rng.standard_normal((n1, Hkv, dh))
    o = O.tree_attention(q, kc, vc, kt, vt, O.tree_mask(spec))
    G = Hq // Hkv
    for i in range(n1):
        path = O.ancestors(spec, i)
        for h in range(Hq):
            g = h // G
            keys = np.concatenate([kc[:, g], kt[path, g]])
            vals = np.concatenate([vc[:, g], vt[path, g]])
            np.testing.assert_allclose(o[i, h], O.attend(q[i, h], keys, vals), rtol=1e-12, atol=1e-14)


def test_single_node_tree_is_plain_decode_attention():
    rng = np.random.default_rng(8)
    spec = O.pack_tree([])
    q = rng.standard_normal((1, 2, 4))
    kc, vc = rng.standard_normal((6, 2, 4)), rng.standard_normal((6, 2, 4))
    kt, vt = rng.standard_normal((1, 2, 4)), rng.standard_normal((1, 2, 4))
    o = O.tree_attention(q, kc, vc, kt, vt, O.tree_mask(spec))
    for h in range(2):
        keys = np.concatenate([kc[:, h], kt[:, h]])
        vals = np.concatenate([vc[:, h], vt[:, h]])
        ref = scipy.special.softmax(keys @ q[0, h] / 2.0) @ vals
        np.testing.assert_allclose(o[0, h], ref, rtol=1e-13)


# ------------------------------------------------------------------ acceptance
def test_entropy_and_threshold_closed_forms():
    V, eps, delta = 1000, 0.09, 0.3
    p = O.softmax_T(np.zeros(V), 0.7)
    assert abs(O.entropy(p) - math.log(V)) < 1e-12
    # uniform: every p = 1/V, threshold min(eps, delta/V) = delta/V > 1/V? no: 0.3/V < 1/V
    ok, _ = O.typical_accept(np.zeros(V), 5, 0.7, eps, delta)
    assert ok == (1.0 / V > min(eps, delta / V))
    # near one-hot: H ~ 0, threshold min(eps, delta) = eps
    z = np.zeros(V)
    z[3] = 200.0
    p = O.softmax_T(z, 1.0)
    assert O.entropy(p) < 1e-60
    assert O.typical_accept(z, 3, 1.0, eps, delta)[0]
    assert not O.typical_accept(z, 4, 1.0, eps, delta)[0]
    # entropy of a two-point distribution against scipy
    z2 = np.full(V, -1e9)
    z2[[1, 2]] = [0.0, math.log(3.0)]
    assert abs(O.entropy(O.softmax_T(z2, 1.0)) - scipy.stats.entropy([0.25, 0.75])) < 1e-12


def test_typical_at_low_temperature_is_greedy():
    """Temperature -> 0 reverts typical acceptance to greedy (Medusa summary §3.4
    'Relationship to temperature')."""
    rng = np.random.default_rng(9)
    for _ in range(30):
        z = rng.standard_normal(300) * 3
        best, margin = O.argmax_lowest(z)
        if margin < 1e-2:
            continue
        for x in [best, (best + 1) % 300, int(rng.integers(300))]:
            ok, _ = O.typical_accept(z, x, 1e-4, 0.09, 0.3)
            assert ok == (x == best)


def _planted_accept_case():
    spec = O.cartesian_tree((2, 2, 2))           # 14 nodes, 8 paths
    n1 = spec.N + 1
    tok = np.arange(100, 100 + n1)
    am = np.full(n1, -1)
    return spec, tok, am


def test_longest_accepted_planted_paths():
    spec, tok, am = _planted_accept_case()
    paths = O.retrieve_paths(spec)
    # plant: path 5 accepted to depth 3, path 1 to depth 2
    target = paths[5]
    for t in range(len(target) - 1):
        am[target[t]] = tok[target[t + 1]]
    p1 = paths[1]
    am[p1[1]] = tok[p1[2]] if am[p1[1]] == -1 else am[p1[1]]
    acc, _ = O.accept_flags(spec, tok, None, am, np.full(len(tok), 1.0), {"mode": "greedy"})
    lens, best, m, nodes = O.longest_accepted(spec, acc)
    assert best == 5 and m == 3 and list(nodes) == target
    # nothing accepted: only the root is kept, the first path wins the tie
    acc0 = np.zeros(spec.N + 1, dtype=np.int64)
    acc0[0] = 1
    lens, best, m, nodes = O.longest_accepted(spec, acc0)
    assert best == 0 and m == 0 and list(nodes) == [0]


def test_longest_accepted_tie_goes_to_lowest_path():
    spec, tok, _ = _planted_accept_case()
    acc = np.zeros(spec.N + 1, dtype=np.int64)
    acc[0] = 1
    paths = O.retrieve_paths(spec)
    for pi in (6, 2):                    # two different depth-2 prefixes
        for n in paths[pi][1:3]:
            acc[n] = 1
    lens, best, m, _ = O.longest_accepted(spec, acc)
    assert m == 2 and best == 2


# ------------------------------------------------------------------ end to end
def _tiny_setup(planted, **over):
    w = S.workload("tiny", **over)
    wts = S.planted_weights(w) if planted else S.weights(w)
    k, v = S.kv_prefix(w, 0)
    ow = O.oracle_weights(wts)
    dims = {"Hq": w.Hq, "Hkv": w.Hkv, "dh": w.dh, "rope_base": w.rope_base}
    return w, ow, S.hidden(w)[0], k, v, dims


@pytest.mark.parametrize("planted", [False, True])
def test_medusa_greedy_reproduces_sequential_greedy(planted):
    """Medusa with greedy verification emits exactly the plain greedy continuation and
    leaves the same KV cache (MEDUSA 精读 section 4: strict greedy verification keeps
    the original model's greedy output)."""
    w, ow, h, k, v, dims = _tiny_setup(planted)
    if planted:
        h = torch.from_numpy(ow["emb"][7].astype(np.float32))   # state of a real token
    spec = O.cartesian_tree(w.s)
    toks, steps, kc, vc = O.medusa_generate(ow, h, k, v, spec, dims, {"mode": "greedy"}, 6)
    ref, kr, vr = O.sequential_greedy(ow, h, k, v, dims, len(toks))
    assert toks == ref
    np.testing.assert_allclose(kc, kr[:len(kc)], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(vc, vr[:len(vc)], rtol=1e-10, atol=1e-12)
    acc_len = [s.m for s in steps]
    if planted:   # the planted model must exercise long and varied paths
        assert np.mean(acc_len) >= 1.0 and max(acc_len) >= 2 and len(set(acc_len)) >= 2
    for s in steps:   # carried root equals the LM head's greedy token at h_next
        assert s.root_next == O.argmax_lowest(O.lm_head(ow["lm"], s.h_next))[0]


def test_typical_temperature_zero_equals_greedy_step():
    w, ow, h, k, v, dims = _tiny_setup(True)
    h = torch.from_numpy(ow["emb"][11].astype(np.float32))
    spec = O.cartesian_tree(w.s)
    g = O.medusa_step(ow, h, k, v, spec, dims, {"mode": "greedy"})
    t = O.medusa_step(ow, h, k, v, spec, dims, {"mode": "typical", "temperature": 0.0,
                                                "eps": 0.09, "delta": 0.3})
    t2 = O.medusa_step(ow, h, k, v, spec, dims, {"mode": "typical", "temperature": 1e-4,
                                                 "eps": 0.09, "delta": 0.3})
    assert list(g.out_tok) == list(t.out_tok) == list(t2.out_tok)
    assert g.m >= 1


def test_step_positions_and_compaction_slots():
    w, ow, h, k, v, dims = _tiny_setup(False)
    spec = O.cartesian_tree(w.s)
    r = O.medusa_step(ow, h, k, v, spec, dims, {"mode": "greedy"})
    assert list(r.pos) == [w.lengths[0] + dd for dd in spec.depth]
    assert len(r.kv_new[0]) == r.m + 1 == len(r.out_tok)
    assert r.out_tok[0] == r.root == O.argmax_lowest(O.lm_head(ow["lm"], O.f64(h)))[0]
    # the kept keys are those of the nodes at depths 0..m on the best path
    assert [spec.depth[n] for n in r.path_nodes] == list(range(r.m + 1))


# ------------------------------------------------------------ rejection sampling (R8)
def _rs_tree():
    """Root with children (0), (1); (0) has children (0,0), (0,1); (1) has child (1,0)."""
    spec = O.pack_tree([[0], [1], [0, 0], [0, 1], [1, 0]])
    tok = np.array([5, 2, 0, 3, 1, 4])          # distinct among siblings, as top-s tokens are
    rng = np.random.default_rng(3)
    zv = rng.standard_normal((spec.N + 1, 6)) * 1.5
    return spec, tok, zv


def test_inverse_cdf_draw_closed_forms():
    w = np.array([0.0, 0.2, 0.0, 0.3, 0.5])
    assert O.inverse_cdf_draw(w, 0.0)[0] == 1           # the first token with weight
    assert O.inverse_cdf_draw(w, 0.5)[0] == 4           # cumulative 0.5 is not > 0.5
    assert O.inverse_cdf_draw(w, 0.49)[0] == 3
    assert O.inverse_cdf_draw(w, 0.999999)[0] == 4
    assert O.inverse_cdf_draw(np.array([0.0, 0.0, 2.0]), 0.7)[0] == 2


def test_rejection_walk_emits_the_backbone_distribution():
    """The speculative-sampling guarantee: the first token after the root is distributed
    as p_root, and the token after an accepted child c as p_c, whatever the drafts."""
    spec, tok, zv = _rs_tree()
    T = 0.9
    n = 40000
    rng = np.random.default_rng(11)
    first = np.zeros(6)
    second = np.zeros(6)
    child = O.children(spec, 0)[0]                      # node (0), token 2
    n_child = 0
    for _ in range(n):
        uni = rng.random(1 + 16 * 2)
        path, v, _ = O.rejection_walk(spec, tok, zv, T, uni)
        t1 = tok[path[1]] if len(path) > 1 else v
        first[t1] += 1
        if len(path) > 1 and path[1] == child:
            n_child += 1
            second[tok[path[2]] if len(path) > 2 else v] += 1
    p0 = O.softmax_T(zv[0], T)
    pc = O.softmax_T(zv[child], T)
    assert n_child > 1000
    for emp, p, m in ((first / n, p0, n), (second / n_child, pc, n_child)):
        sigma = np.sqrt(p * (1 - p) / m)
        assert (np.abs(emp - p) < 5 * sigma + 1e-12).all(), (emp, p)


def test_rejection_walk_at_low_temperature_is_the_greedy_walk():
    spec, tok, zv = _rs_tree()
    tok = tok.copy()                                    # plant greedy matches along (0), (0,1)
    tok[1] = int(np.argmax(zv[0]))                      # child (0) is the root's greedy token
    tok[2] = (tok[1] + 1) % 6
    tok[4] = int(np.argmax(zv[1]))                      # child (0,1) is (0)'s greedy token
    tok[3] = (tok[4] + 1) % 6
    rng = np.random.default_rng(5)
    am = np.array([int(np.argmax(z)) for z in zv])
    acc, _ = O.accept_flags(spec, tok, zv, am, np.full(spec.N + 1, np.inf), {"mode": "greedy"})
    _, _, m, greedy_path = O.longest_accepted(spec, acc)
    for _ in range(20):
        path, v, _ = O.rejection_walk(spec, tok, zv, 1e-4, rng.random(1 + 32) * 0.999 + 0.0005)
        assert list(path) == list(greedy_path)
        assert v == am[path[-1]]


# ---------------------------------------------------------------- multi-layer backbone (R14)
def _layers_setup(planted, n_layers):
    w, ow, h, k, v, dims = _tiny_setup(planted)
    layers = [ow] + [O.oracle_weights(S.layer_weights(w, l, planted=planted))
                     for l in range(1, n_layers)]
    caches = [(k, v)] + [S.kv_prefix(w, 0, l) for l in range(1, n_layers)]
    return w, ow, h, layers, caches, dims


def test_one_layer_backbone_is_the_single_layer_step():
    """R14 with one layer is R0: the same tokens, layer outputs, logits and path."""
    w, ow, h, layers, caches, dims = _layers_setup(True, 1)
    h = torch.from_numpy(ow["emb"][7].astype(np.float32))
    spec = O.cartesian_tree(w.s)
    a = O.medusa_step(ow, h, caches[0][0], caches[0][1], spec, dims, {"mode": "greedy"})
    b = O.medusa_step_layers(ow, layers, h, caches, spec, dims, {"mode": "greedy"})
    assert list(a.tok) == list(b.tok) and list(a.path_nodes) == list(b.path_nodes)
    np.testing.assert_array_equal(a.hp, b.hp)
    np.testing.assert_array_equal(a.zv, b.zv)
    np.testing.assert_array_equal(a.kv_new[0], b.kv_new_layers[0][0])


def test_layers_differ_so_the_pins_below_see_every_layer():
    """Layer 1's projections and cache are not layer 0's, and a second layer changes
    h' (a dropped layer loop or a reused cache would fail the decoding pins)."""
    w, ow, h, layers, caches, dims = _layers_setup(False, 2)
    assert not np.array_equal(layers[0]["wq"], layers[1]["wq"])
    assert not np.array_equal(O.f64(caches[0][0]), O.f64(caches[1][0]))
    spec = O.cartesian_tree(w.s)
    one = O.medusa_step_layers(ow, layers[:1], h, caches[:1], spec, dims, {"mode": "greedy"})
    two = O.medusa_step_layers(ow, layers, h, caches, spec, dims, {"mode": "greedy"})
    assert np.abs(one.hp - two.hp).max() > 1e-3
    np.testing.assert_array_equal(one.layer_k[0], two.layer_k[0])   # layer 0 sees layer 0 only


@pytest.mark.parametrize("planted,n_layers", [(False, 2), (True, 3)])
def test_multi_layer_medusa_greedy_reproduces_sequential_greedy(planted, n_layers):
    """Through an n-layer backbone, Medusa with greedy verification emits the plain greedy
    continuation and leaves every layer's cache as sequential decoding does (MEDUSA 精读
    section 4), so tree attention and compaction are right in every layer."""
    w, ow, h, layers, caches, dims = _layers_setup(planted, n_layers)
    if planted:
        h = torch.from_numpy(ow["emb"][7].astype(np.float32))
    spec = O.cartesian_tree(w.s)
    toks, steps, fin = O.medusa_generate_layers(ow, layers, h, caches, spec, dims,
                                                {"mode": "greedy"}, 5)
    ref, ref_caches = O.sequential_greedy_layers(ow, layers, h, caches, dims, len(toks))
    assert toks == ref
    for (kc, vc), (kr, vr) in zip(fin, ref_caches):
        np.testing.assert_allclose(kc, kr[:len(kc)], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(vc, vr[:len(vc)], rtol=1e-10, atol=1e-12)
    if planted:
        assert max(s.m for s in steps) >= 2


def test_verify_only_equals_the_steps_verification():
    """verify_only on a step's own layer outputs and tokens reproduces that step's
    acceptance, path, next root and hidden state."""
    w = S.workload("tiny", mode="typical", temperature=0.7)
    wts = S.weights(w)
    ow = O.oracle_weights(wts)
    spec = O.cartesian_tree(w.s)
    k, v = S.kv_prefix(w, 0)
    dims = {"Hq": w.Hq, "Hkv": w.Hkv, "dh": w.dh, "rope_base": w.rope_base}
    acc = {"mode": "typical", "temperature": 0.7, "eps": w.eps, "delta": w.delta}
    r = O.medusa_step(ow, S.hidden(w)[0], k, v, spec, dims, acc, s=list(w.s))
    q = O.verify_only(ow, r.hp, r.tok, spec, acc)
    assert list(q.acc) == list(r.acc) and list(q.path_nodes) == list(r.path_nodes)
    assert q.root_next == r.root_next and np.array_equal(q.h_next, r.h_next)
    np.testing.assert_array_equal(q.zv, r.zv)
