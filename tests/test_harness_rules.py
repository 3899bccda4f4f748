"""The parity harness's comparison rules, checked on the CPU: a 'GPU' output made from the
oracle's own step passes; a planted mismatch fails unless the one decision it changes is a
near tie (oracle margin below 1e-3), and a near tie excuses only that decision, not a
mismatch elsewhere in the same sequence.  Mistakes are planted in copies of the oracle's
results; nothing here runs the library."""
import copy

import numpy as np
import pytest

import oracle as O
import synthetic as S
from harness import Flagged, compare_sequence

W = S.workload("tiny")


def _oracle_result(mode="greedy", T=0.0):
    wts = S.weights(W)
    ow = O.oracle_weights(wts)
    spec = O.cartesian_tree(W.s)
    k, v = S.kv_prefix(W, 0)
    dims = {"Hq": W.Hq, "Hkv": W.Hkv, "dh": W.dh, "rope_base": W.rope_base}
    acc = {"mode": mode, "temperature": T, "eps": W.eps, "delta": W.delta}
    r = O.medusa_step(ow, S.hidden(W)[0], k, v, spec, dims, acc, s=list(W.s))
    return r, spec


def _fake_gpu(r, spec, T=0.0):
    """Stage outputs laid out as the library returns them, holding the oracle's values."""
    n1, K = spec.N + 1, W.K
    g = {}
    g["logits"] = np.concatenate([r.z0[None], r.zk])[None].astype(np.float32)
    tt = np.full((1, K, 16), -1, np.int32)
    tt[0, :, :r.topk.shape[1]] = r.topk
    g["topk_tok"] = tt
    g["root"] = np.array([r.root], np.int32)
    g["tok"] = r.tok[None].astype(np.int32)
    g["pos"] = r.pos[None].astype(np.int32)
    M = O.tree_mask(spec)
    bits = np.zeros((n1, 8), np.uint32)
    for i in range(n1):
        for j in range(n1):
            if M[i, j]:
                bits[i, j // 32] |= np.uint32(1 << (j % 32))
    g["mask"] = bits.view(np.int32)
    retr = np.full((n1, K + 1), -1, np.int32)
    for pi, p in enumerate(O.retrieve_paths(spec)):
        retr[pi, :len(p)] = p
    g["retrieve"] = retr
    for name, x in (("q", r.q), ("tk", r.k), ("tv", r.v), ("o", r.o), ("hp", r.hp), ("vlog", r.zv)):
        g[name] = x[None].astype(np.float32)
    g["am"] = r.am[None].astype(np.int32)
    st = np.zeros((1, n1, 4), np.float32)
    Tn = T if T > 0 else 1.0
    for n in range(n1):
        z = r.zv[n] / Tn
        mx = z.max()
        p = np.exp(z - mx)
        st[0, n, 0], st[0, n, 1] = mx, np.log(p.sum())
        p /= p.sum()
        st[0, n, 2] = -(p[p > 0] * np.log(p[p > 0])).sum()
        if n > 0:
            st[0, n, 3] = r.zv[spec.parent[n], r.tok[n]] / Tn
    g["stats"] = st
    _set_path(g, r.path_nodes)
    g["root_next"] = np.array([r.root_next], np.int32)
    return g


def _set_path(g, nodes):
    K = W.K
    nodes = [int(x) for x in nodes]
    g["n_acc"] = np.array([len(nodes)], np.int32)
    g["path"] = np.full((1, K + 1), -1, np.int32)
    g["path"][0, :len(nodes)] = nodes
    g["out_tok"] = np.full((1, K + 1), -1, np.int32)
    g["out_tok"][0, :len(nodes)] = g["tok"][0, nodes]
    g["h_next"] = g["hp"][0, nodes[-1]][None].copy()
    g["root_next"] = np.array([g["am"][0, nodes[-1]]], np.int32)


def _greedy_path(g, spec):
    acc = np.zeros(spec.N + 1, np.int64)
    acc[0] = 1
    for c in range(1, spec.N + 1):
        acc[c] = int(g["tok"][0, c] == g["am"][0, spec.parent[c]])
    return O.longest_accepted(spec, acc)[3]


def test_exact_outputs_pass():
    r, spec = _oracle_result()
    compare_sequence(_fake_gpu(r, spec), r, 0, spec, W, {})


def test_typical_exact_outputs_pass():
    w = S.workload("tiny", mode="typical", temperature=0.7)
    r, spec = _oracle_result("typical", 0.7)
    compare_sequence(_fake_gpu(r, spec, 0.7), r, 0, spec, w, {})


def test_argmax_mismatch_away_from_a_tie_fails():
    r, spec = _oracle_result()
    g = _fake_gpu(r, spec)
    c = 1                                   # make the root's greedy token node 1's token
    g["am"][0, 0] = g["tok"][0, c]
    _set_path(g, _greedy_path(g, spec))
    r.am_margin[0] = 0.5
    r.acc_margin[[n for n in range(1, spec.N + 1) if spec.parent[n] == 0]] = 0.5
    with pytest.raises(AssertionError):
        compare_sequence(g, r, 0, spec, W, {})


def test_near_tie_at_the_differing_node_is_flagged():
    r, spec = _oracle_result()
    g = _fake_gpu(r, spec)
    c = 1
    g["am"][0, 0] = g["tok"][0, c]          # the GPU's root argmax picks node 1's token
    _set_path(g, _greedy_path(g, spec))
    assert g["n_acc"][0] >= 2
    r.am_margin[0] = 1e-4                   # ... where the oracle's top-2 gap is a near tie
    for n in range(1, spec.N + 1):
        if spec.parent[n] == 0:
            r.acc_margin[n] = 1e-4
    with pytest.raises(Flagged):
        compare_sequence(g, r, 0, spec, W, {})


def test_near_tie_elsewhere_does_not_excuse_a_mismatch():
    r, spec = _oracle_result()
    g = _fake_gpu(r, spec)
    # a near tie at a node the GPU agrees on ...
    far = spec.N
    r.am_margin[far] = 1e-4
    r.acc_margin[[n for n in range(1, spec.N + 1) if spec.parent[n] == far]] = 1e-4
    # ... and a real difference at the root's decision
    g["am"][0, 0] = g["tok"][0, 1]
    _set_path(g, _greedy_path(g, spec))
    r.am_margin[0] = 0.5
    r.acc_margin[[n for n in range(1, spec.N + 1) if spec.parent[n] == 0]] = 0.5
    with pytest.raises(AssertionError):
        compare_sequence(g, r, 0, spec, W, {})


def test_wrong_path_choice_fails():
    r, spec = _oracle_result()
    g = _fake_gpu(r, spec)
    # every flag as the oracle's, but a path that is not the longest accepted prefix
    _set_path(g, [0, spec.N - 1] if spec.parent[spec.N - 1] == 0 else [0, 1])
    with pytest.raises(AssertionError):
        compare_sequence(g, r, 0, spec, W, {})


def test_near_tie_top_s_swap_leaves_the_rest_compared():
    r, spec = _oracle_result()
    g = _fake_gpu(r, spec)
    k, a, b = 0, 1, 2                        # swap head 1's ranks 1 and 2 on the 'GPU'
    tt = g["topk_tok"]
    tt[0, k, a], tt[0, k, b] = tt[0, k, b], tt[0, k, a]
    for n in range(1, spec.N + 1):
        if spec.depth[n] == 1 and spec.rank[n] in (a, b):
            g["tok"][0, n] = tt[0, k, spec.rank[n]]
    r.topk_margin[k, a] = r.topk_margin[k, b] = 1e-4
    _set_path(g, _greedy_path(g, spec))
    with pytest.raises(Flagged):
        compare_sequence(g, r, 0, spec, W, {})
    # an attention error at a node outside the swapped subtrees is still caught
    g2 = copy.deepcopy(g)
    g2["o"][0, 0, 0, 0] += 1.0
    with pytest.raises(AssertionError):
        compare_sequence(g2, r, 0, spec, W, {})


def _typical_flip():
    """Typical mode: the 'GPU' statistics accept node 1 where the oracle rejects it."""
    w = S.workload("tiny", mode="typical", temperature=0.7)
    r, spec = _oracle_result("typical", 0.7)
    g = _fake_gpu(r, spec, 0.7)
    c = next(n for n in range(1, spec.N + 1) if not r.acc[n] and spec.parent[n] == 0)
    g["stats"][0, c, 3] = g["stats"][0, 0, 0]            # p_root(tok_c) -> the maximum
    acc = np.zeros(spec.N + 1, np.int64)
    acc[0] = 1
    st = g["stats"][0]
    for n in range(1, spec.N + 1):
        p = spec.parent[n]
        lp = st[n, 3] - st[p, 0] - st[p, 1]
        acc[n] = int(lp > min(np.log(w.eps), np.log(w.delta) - st[p, 2]))
    _set_path(g, O.longest_accepted(spec, acc)[3])
    return w, r, spec, g, c


def test_typical_accept_flag_mismatch_fails():
    w, r, spec, g, c = _typical_flip()
    r.acc_margin[c] = 0.5
    with pytest.raises(AssertionError, match="accept flag"):
        compare_sequence(g, r, 0, spec, w, {})


def test_typical_accept_flag_near_tie_is_flagged():
    w, r, spec, g, c = _typical_flip()
    r.acc_margin[c] = 1e-4
    with pytest.raises(Flagged, match=f"accept node {c}"):
        compare_sequence(g, r, 0, spec, w, {})
