"""Verification alone on seeded logits (the 13B configuration's "fixed-seed logits"):
the layer outputs h' are drawn directly and the LM head is the identity (d = V), so the
verification logits are the drawn values themselves, up to the bf16 hi/lo split of h'
(~2^-17 relative) and no other GEMM rounding.  Node tokens are planted so that a chosen
share of the candidates is accepted, and for typical acceptance some candidates are
planted close to (but outside) the 1e-3 flag window of the threshold.  medusa_verify_logits
then medusa_verify must take exactly the oracle's decisions, path and outputs."""
import numpy as np
import pytest
import torch

import oracle as O
import synthetic as S
from medusa_head_speculative_gb300 import binding as Bnd

from harness import NEAR, ensure_built, gpu_accept_flags, record, spec_for

pytestmark = pytest.mark.gpu


def _workload(mode, T, B=4):
    return S.Workload(name=f"seeded_{mode}", B=B, d=1024, V=1024, Hq=4, Hkv=4, dh=64, K=4,
                      dtype="bf16", lengths=(16,) * B, tree="greedy", s=(10,) * 4, N=40,
                      mode=mode, temperature=T)


def _plant_near(z, p, x, accept, target, rng):
    """Move logit z[p][x] so that the oracle's typical decision for token x at node p sits
    `target` (signed, in log units) from the threshold; returns the margin reached."""
    T, eps, delta = accept["temperature"], accept["eps"], accept["delta"]

    def signed(v):
        zz = z[p].astype(np.float64).copy()
        zz[x] = v
        pr = O.softmax_T(zz, T)
        thr = min(eps, delta * np.exp(-O.entropy(pr)))
        return np.log(pr[x]) - np.log(thr)

    lo, hi = -40.0, 40.0
    for _ in range(80):                        # signed() increases with the logit
        mid = 0.5 * (lo + hi)
        if signed(mid) < target:
            lo = mid
        else:
            hi = mid
    z[p, x] = np.float32(0.5 * (lo + hi))
    return signed(float(z[p, x]))


def _inputs(w, spec, accept, p_accept, seed):
    rng = np.random.default_rng(seed)
    n1 = spec.N + 1
    sigma = 2.0
    z = (rng.standard_normal((w.B, n1, w.V)) * sigma).astype(np.float32)
    tok = rng.integers(0, w.V, size=(w.B, n1)).astype(np.int32)
    near = 0
    for b in range(w.B):
        for c in range(1, n1):
            p = spec.parent[c]
            u = rng.random()
            if u < p_accept:                                   # the parent's greedy token
                tok[b, c] = int(np.argmax(z[b, p]))
            elif u < p_accept + 0.25:                          # one of its next few
                tok[b, c] = int(np.argsort(-z[b, p])[rng.integers(1, 6)])
        if accept["mode"] == "typical":
            # near-threshold candidates, 2e-3 .. 1e-2 from the boundary on either side (one
            # per parent: moving a logit moves the parent's entropy for all its children)
            used = set()
            for c in rng.choice(np.arange(1, n1), size=8, replace=False):
                p = spec.parent[c]
                if p in used or any(spec.parent[o] == p and o != c and tok[b, o] == tok[b, c]
                                    for o in range(1, n1)):
                    continue
                used.add(p)
                target = rng.choice([-1.0, 1.0]) * rng.uniform(2e-3, 1e-2)
                m = _plant_near(z[b], p, int(tok[b, c]), accept, target, rng)
                near += abs(m) < 2e-2
    return z, tok, near


@pytest.mark.parametrize("mode,T,p_accept", [("greedy", 0.0, 0.6), ("typical", 0.7, 0.4),
                                             ("typical", 1.0, 0.2)])
def test_verify_on_seeded_logits_matches_oracle(mode, T, p_accept):
    ensure_built()
    w = _workload(mode, T)
    parent, rank, spec = spec_for(w)
    plan = Bnd.Plan(w.B, w.d, w.V, w.K, w.Hq, w.Hkv, w.dh, Bnd.BF16, w.capacity, w.s, parent,
                    rank, rope_base=w.rope_base)
    accept = {"mode": mode, "temperature": T, "eps": w.eps, "delta": w.delta}
    z, tok, near = _inputs(w, spec, accept, p_accept, seed=17 + int(10 * T))
    lm = torch.eye(w.V, w.d, dtype=torch.bfloat16)           # logits = h' exactly
    n1 = spec.N + 1
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    hp, tk = dev(z), dev(tok)
    wst = Bnd.weights_struct({"lm": lm.cuda()})
    ws = torch.empty(plan.workspace_size, dtype=torch.uint8, device="cuda")
    acc = Bnd.accept_struct(mode, T, w.eps, w.delta)
    i32, f32 = dict(dtype=torch.int32, device="cuda"), dict(dtype=torch.float32, device="cuda")
    vlog = torch.empty(w.B, n1, w.V, **f32)
    am = torch.empty(w.B, n1, **i32)
    stats = torch.empty(w.B, n1, 4, **f32)
    Bnd.verify_logits(plan, wst, hp, tk, acc, vlog, am, stats, ws)
    # the library's own root->leaf table, from a tree build on any valid candidates
    ttok = torch.zeros(w.B, w.K, 16, **i32)
    root = torch.zeros(w.B, **i32)
    retr = torch.empty(n1, w.K + 1, **i32)
    Bnd.tree_build(plan, ttok, root, torch.full((w.B,), 16, **i32), torch.empty(w.B, n1, **i32),
                   torch.empty(w.B, n1, **i32), torch.empty(n1, 8, **i32), retr)
    out_tok = torch.empty(w.B, w.K + 1, **i32)
    n_acc = torch.empty(w.B, **i32)
    path = torch.empty(w.B, w.K + 1, **i32)
    h_next = torch.empty(w.B, w.d, **f32)
    root_next = torch.empty(w.B, **i32)
    outs = Bnd.outputs_struct(out_tok, n_acc, path, h_next, root_next)
    Bnd.verify(plan, tk, am, stats, retr, hp, acc, outs, logits=vlog)
    torch.cuda.synchronize()
    assert plan.status() == 0
    g = {"tok": tok, "am": am.cpu().numpy(), "stats": stats.cpu().numpy()}
    np.testing.assert_allclose(vlog.cpu().numpy(), z, rtol=2e-5, atol=1e-5)
    ow = {"lm": np.eye(w.V, w.d)}
    accepted, compared, flagged = 0, 0, []
    for b in range(w.B):
        r = O.verify_only(ow, z[b], tok[b], spec, accept)
        differs = False
        for n in range(n1):
            if g["am"][b, n] != r.am[n]:
                assert r.am_margin[n] < NEAR, (b, n)
                differs = True
        gacc, amb = gpu_accept_flags(g, b, spec, w)
        for c in range(1, n1):
            if gacc[c] != r.acc[c]:
                assert r.acc_margin[c] < NEAR or amb[c], (b, c, r.acc_margin[c])
                differs = True
        if differs:
            flagged.append((b, "near-tie decision"))
            continue
        compared += 1
        m = int(n_acc[b]) - 1
        assert m == r.m
        assert list(path[b, :m + 1].cpu().numpy()) == list(r.path_nodes)
        assert list(out_tok[b, :m + 1].cpu().numpy()) == list(r.out_tok)
        assert int(root_next[b]) == r.root_next
        np.testing.assert_array_equal(h_next[b].cpu().numpy(), z[b, r.path_nodes[-1]])
        accepted += int(r.acc[1:].sum())
    record(f"verify_seeded_{mode}_{T}", compared, flagged)
    assert compared >= w.B - 1
    assert accepted >= 0.1 * w.B * spec.N                     # the planted share is accepted
    if mode == "typical":
        assert near >= w.B                                    # near-threshold cases were planted
