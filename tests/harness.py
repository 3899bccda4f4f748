"""Helpers of the GPU parity tests: set up a workload on the device, run the library's
stages through the C ABI, run the oracle on the same seeded inputs, and compare under
the stated rules:

* indices, tree tables, tokens and accepted paths bit-exact;
* a decision whose fp64 oracle margin is below 1e-3 (top-2 logit gap, top-s neighbour
  gap, |log p - log threshold|) is flagged, not failed, when it comes out differently on
  the GPU: only that decision is excused, the outputs that depend on it are left out and
  everything else of the sequence is still compared; the sequence then counts as
  flagged, and each case states how many flagged sequences it allows;
* floats (logits, q/k/v, attention outputs, h', cache rows) within |gpu - oracle| <=
  2e-2 + 1e-2 |oracle|.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

import oracle as O
import synthetic as S
from medusa_head_speculative_gb300 import binding as Bnd

ATOL, RTOL = 2e-2, 1e-2
NEAR = O.NEAR


def ensure_built():
    import os
    if not os.path.exists(Bnd.LIB_PATH):
        from medusa_head_speculative_gb300 import build
        build.build()
    Bnd.lib()


def close(g, o, atol=ATOL, rtol=RTOL):
    g = np.asarray(g, dtype=np.float64)
    o = np.asarray(o, dtype=np.float64)
    assert g.shape == o.shape, (g.shape, o.shape)
    err = np.abs(g - o) - (atol + rtol * np.abs(o))
    return float(err.max()) if err.size else -1.0


def spec_for(w: S.Workload):
    """(product-built parent/rank, oracle-built TreeSpec); asserted equal."""
    if w.tree == "cartesian":
        parent, rank = Bnd.tree_cartesian(w.s)
        spec = O.cartesian_tree(w.s)
    else:
        a = S.score_table(w.K, max(w.s))
        parent, rank = Bnd.tree_greedy(w.s, a, w.N)
        spec = O.greedy_tree(a, w.s, w.N)
    assert list(parent) == spec.parent and list(rank) == spec.rank
    return parent, rank, spec


@dataclass
class Device:
    w: S.Workload
    plan: Bnd.Plan
    wts: dict
    wstruct: object
    h: torch.Tensor
    kc: torch.Tensor
    vc: torch.Tensor
    pt: torch.Tensor
    length: torch.Tensor
    ws: torch.Tensor
    spec: O.TreeSpec
    cpu: dict = field(default_factory=dict)
    uni: torch.Tensor = None          # rejection sampling: device uniforms [B][1 + 16 K]


def setup(w: S.Workload, wts_cpu=None, h_cpu=None, host_seqs=None):
    """The workload on the device.  host_seqs: only these sequences' KV prefixes come from
    the host streams (the oracle's inputs); the others are drawn on the device."""
    ensure_built()
    parent, rank, spec = spec_for(w)
    dtype = Bnd.F32 if w.dtype == "f32" else Bnd.BF16
    num_pages = w.B * w.pages_per_seq if w.page_size else 0
    plan = Bnd.Plan(w.B, w.d, w.V, w.K, w.Hq, w.Hkv, w.dh, dtype, w.capacity, w.s, parent, rank,
                    rope_base=w.rope_base, page_size=w.page_size, num_pages=num_pages)
    wts_cpu = wts_cpu if wts_cpu is not None else S.weights(w)
    wts = {k: v.cuda() for k, v in wts_cpu.items()}
    h_cpu = h_cpu if h_cpu is not None else S.hidden(w)
    if host_seqs is None:
        kc, vc, pt = S.kv_cache(w)
        kc, vc, pt = kc.cuda(), vc.cuda(), None if pt is None else pt.cuda()
    else:
        kc, vc, pt = S.kv_cache_device(w, host_seqs, torch.device("cuda"))
    dev = Device(w, plan, wts, Bnd.weights_struct(wts), h_cpu.cuda(), kc, vc, pt,
                 torch.tensor(w.lengths, dtype=torch.int32, device="cuda"),
                 torch.empty(plan.workspace_size, dtype=torch.uint8, device="cuda"), spec)
    dev.cpu = {"wts": wts_cpu, "h": h_cpu}
    if w.mode == "reject":
        dev.uni = S.uniforms(w).cuda()
    return dev


def accept_of(w: S.Workload, dev=None):
    """Acceptance parameters for the binding (dev given: with the device uniforms of a
    rejection-sampling workload)."""
    a = {"mode": w.mode, "temperature": w.temperature, "eps": w.eps, "delta": w.delta}
    if w.mode == "reject" and dev is not None:
        a["uniforms"] = dev.uni
    return a


def oracle_accept(w: S.Workload, b: int):
    """The same parameters for the oracle's sequence b."""
    a = {"mode": w.mode, "temperature": w.temperature, "eps": w.eps, "delta": w.delta}
    if w.mode == "reject":
        a["uniforms"] = S.uniforms(w)[b].numpy().astype(np.float64)
    return a


def run_stages(dev: Device, root_in=None):
    """Every stage through its own entry point, chained on the GPU; returns CPU copies."""
    w, p = dev.w, dev.plan
    B, K, V, d, n1 = w.B, w.K, w.V, w.d, p.n1
    f32, i32 = dict(dtype=torch.float32, device="cuda"), dict(dtype=torch.int32, device="cuda")
    kvdt = dict(dtype=w.torch_dtype, device="cuda")
    r = {}
    logits = torch.empty(B, K + 1, V, **f32)
    ttok = torch.empty(B, K, 16, **i32)
    tval = torch.empty(B, K, 16, **f32)
    root = torch.empty(B, **i32)
    Bnd.heads(p, dev.h, root_in, dev.wstruct, logits, ttok, tval, root, dev.ws)
    tok = torch.empty(B, n1, **i32)
    pos = torch.empty(B, n1, **i32)
    mask = torch.empty(n1, 8, dtype=torch.int32, device="cuda")
    retr = torch.empty(n1, K + 1, **i32)
    Bnd.tree_build(p, ttok, root, dev.length, tok, pos, mask, retr)
    q = torch.empty(B, n1, w.Hq, w.dh, **f32)
    tk = torch.empty(B, n1, w.Hkv, w.dh, **kvdt)
    tv = torch.empty(B, n1, w.Hkv, w.dh, **kvdt)
    Bnd.layer_qkv(p, dev.wstruct, tok, pos, q, tk, tv, dev.ws)
    kv = Bnd.kv_struct(dev.kc, dev.vc, dev.length, None, dev.pt)
    o = torch.empty(B, n1, w.Hq, w.dh, **f32)
    Bnd.tree_attention(p, q, kv, tk, tv, mask, o, dev.ws)
    hp = torch.empty(B, n1, d, **f32)
    Bnd.layer_out(p, dev.wstruct, tok, o, hp, dev.ws)
    acc = Bnd.accept_struct(**accept_of(w, dev))
    vlog = torch.empty(B, n1, V, **f32)
    am = torch.empty(B, n1, **i32)
    stats = torch.empty(B, n1, 4, **f32)
    Bnd.verify_logits(p, dev.wstruct, hp, tok, acc, vlog, am, stats, dev.ws)
    out_tok = torch.empty(B, K + 1, **i32)
    n_acc = torch.empty(B, **i32)
    path = torch.empty(B, K + 1, **i32)
    h_next = torch.empty(B, d, **f32)
    root_next = torch.empty(B, **i32)
    outs = Bnd.outputs_struct(out_tok, n_acc, path, h_next, root_next)
    Bnd.verify(p, tok, am, stats, retr, hp, acc, outs, logits=vlog)
    torch.cuda.synchronize()
    for name, t in [("logits", logits), ("topk_tok", ttok), ("topk_val", tval), ("root", root),
                    ("tok", tok), ("pos", pos), ("mask", mask), ("retrieve", retr), ("q", q),
                    ("tk", tk), ("tv", tv), ("o", o), ("hp", hp), ("vlog", vlog), ("am", am),
                    ("stats", stats), ("out_tok", out_tok), ("n_acc", n_acc), ("path", path),
                    ("h_next", h_next), ("root_next", root_next)]:
        r[name] = t.float().cpu().numpy() if t.dtype == torch.bfloat16 else t.cpu().numpy()
    r["_dev"] = dict(tk=tk, tv=tv, path=path, n_acc=n_acc)
    return r


def run_step(dev: Device, root_in=None, len_out=None):
    """One medusa_step; the cache is updated in place, lengths into len_out (or in place)."""
    w, p = dev.w, dev.plan
    B, K, d = w.B, w.K, w.d
    i32 = dict(dtype=torch.int32, device="cuda")
    out_tok = torch.empty(B, K + 1, **i32)
    n_acc = torch.empty(B, **i32)
    path = torch.empty(B, K + 1, **i32)
    h_next = torch.empty(B, d, dtype=torch.float32, device="cuda")
    root_next = torch.empty(B, **i32)
    len_out = dev.length if len_out is None else len_out
    kv = Bnd.kv_struct(dev.kc, dev.vc, dev.length, len_out, dev.pt)
    outs = Bnd.outputs_struct(out_tok, n_acc, path, h_next, root_next)
    Bnd.step(p, dev.h, root_in, dev.wstruct, kv, Bnd.accept_struct(**accept_of(w, dev)), outs, dev.ws)
    torch.cuda.synchronize()
    return dict(out_tok=out_tok.cpu().numpy(), n_acc=n_acc.cpu().numpy(), path=path.cpu().numpy(),
                h_next=h_next, root_next=root_next, len_out=len_out.cpu().numpy())


def oracle_step(dev: Device, b: int, ow=None, root=None):
    w = dev.w
    ow = ow if ow is not None else O.oracle_weights(dev.cpu["wts"])
    k, v = S.kv_prefix(w, b)
    dims = {"Hq": w.Hq, "Hkv": w.Hkv, "dh": w.dh, "rope_base": w.rope_base}
    return O.medusa_step(ow, dev.cpu["h"][b], k, v, dev.spec, dims, oracle_accept(w, b), root=root,
                         s=list(w.s))


class Flagged(Exception):
    """A near-tie decision (oracle margin below NEAR) came out differently on the GPU.
    Raised only after every output that does not depend on it has been compared."""


def affected_nodes(spec: O.TreeSpec, bad_ranks) -> np.ndarray:
    """Nodes whose token comes from a top-s rank in `bad_ranks` ({(head index k, rank)}),
    and all their descendants (their attention reads those nodes' keys and values)."""
    n1 = spec.N + 1
    aff = np.zeros(n1, dtype=bool)
    for n in range(1, n1):
        d = spec.depth[n]
        aff[n] = (d - 1, spec.rank[n]) in bad_ranks or aff[spec.parent[n]]
    return aff


def gpu_accept_flags(g: dict, b: int, spec: O.TreeSpec, w: S.Workload):
    """The GPU's accept flag of every node, recomputed from its own outputs (node tokens,
    per-node greedy tokens and statistics) by the rule the library documents for
    medusa_verify, in fp32 as the kernel evaluates it.  Returns (acc, ambiguous): ambiguous
    marks typical decisions within fp32 rounding of the threshold, where this recomputation
    cannot tell which way the kernel went."""
    n1 = spec.N + 1
    acc = np.zeros(n1, dtype=np.int64)
    amb = np.zeros(n1, dtype=bool)
    acc[0] = 1
    typical = w.mode == "typical" and w.temperature > 0
    st = g["stats"][b].astype(np.float32)
    tok, am = g["tok"][b], g["am"][b]
    le = np.log(np.float32(w.eps), dtype=np.float32)
    ld = np.log(np.float32(w.delta), dtype=np.float32)
    for c in range(1, n1):
        p = spec.parent[c]
        if typical:
            lp = np.float32(np.float32(st[c, 3] - st[p, 0]) - st[p, 1])
            thr = min(le, np.float32(ld - st[p, 2]))
            acc[c] = int(lp > thr)
            amb[c] = abs(float(lp) - float(thr)) <= 1e-5 * max(1.0, abs(float(thr)))
        else:
            acc[c] = int(tok[c] == am[p])
    return acc, amb


def explain_by_flips(spec: O.TreeSpec, r: O.StepResult, g_path, excusable) -> bool:
    """True when the GPU's kept path g_path (packed node indices root..last) is what the
    longest-path rule gives for accept flags that differ from the oracle's only at nodes
    in `excusable`.  The flags most favourable to g_path are used: excusable nodes on
    g_path accepted, every other excusable node rejected."""
    acc = np.array(r.acc, dtype=np.int64).copy()
    acc[excusable] = 0
    acc[list(g_path)] = 1
    _, _, m, nodes = O.longest_accepted(spec, acc)
    return m == len(g_path) - 1 and list(nodes) == list(g_path)


def compare_sequence(g: dict, r: O.StepResult, b: int, spec: O.TreeSpec, w: S.Workload,
                     report: dict, root_given: bool = False):
    """Compare GPU stage outputs of sequence b with the oracle's step.

    Raises AssertionError on a real mismatch.  A decision whose oracle margin is below
    NEAR and that came out differently on the GPU is excused, but only that decision:
    the outputs that depend on it (the subtree of a swapped top-s rank, the children of
    a node whose greedy token differs, the path once an accept flag differs) are left
    out and everything else is compared.  Flagged is raised at the end when anything was
    excused.  With root_given the LM head's logits on h_t are not computed on the GPU
    and not compared."""
    K, n1 = w.K, spec.N + 1
    report.setdefault("near_ties", 0)
    excused = []
    # heads
    if not root_given:
        assert close(g["logits"][b, 0], r.z0) <= 0, "LM-head logits"
    assert close(g["logits"][b, 1:], r.zk) <= 0, "head logits"
    bad_ranks = set()
    for k in range(K):
        for rk in range(w.s[k]):
            if r.topk_margin[k, rk] < NEAR:
                report["near_ties"] += 1
            if g["topk_tok"][b, k, rk] != r.topk[k, rk]:
                if r.topk_margin[k, rk] < NEAR:
                    excused.append(f"top-s head {k + 1} rank {rk}")
                    bad_ranks.add((k, rk))
                    continue
                raise AssertionError(f"top-s head {k + 1} rank {rk}: {g['topk_tok'][b, k, rk]} "
                                     f"!= {r.topk[k, rk]}")
    if g["root"][b] != r.root:
        if r.root_margin < NEAR:           # every node attends to the root: nothing further
            raise Flagged("root")
        raise AssertionError(f"root {g['root'][b]} != {r.root}")
    # tree tables (independent of the tokens)
    assert (g["pos"][b] == r.pos).all(), "positions"
    M = O.tree_mask(spec)
    bits = g["mask"].view(np.uint32)
    for i in range(n1):
        for j in range(n1):
            assert ((bits[i, j // 32] >> (j % 32)) & 1) == M[i, j], f"mask {i},{j}"
        for j in range(n1, 256):
            assert ((bits[i, j // 32] >> (j % 32)) & 1) == 0
    paths = O.retrieve_paths(spec)
    for pi, path in enumerate(paths):
        assert list(g["retrieve"][pi, :len(path)]) == path
        assert (g["retrieve"][pi, len(path):] == -1).all()
    assert (g["retrieve"][len(paths):] == -1).all()
    # node tokens: the oracle's where no excused rank reaches, else the GPU's own top-s
    aff = affected_nodes(spec, bad_ranks)
    ok = ~aff
    for n in range(n1):
        if ok[n]:
            assert g["tok"][b, n] == r.tok[n], f"node {n} token"
        else:
            assert g["tok"][b, n] == g["topk_tok"][b, spec.depth[n] - 1, spec.rank[n]]
    # synthetic layer, attention, h' and verification logits of the unaffected nodes
    assert close(g["q"][b][ok], r.q[ok]) <= 0, "q"
    assert close(g["tk"][b][ok], r.k[ok]) <= 0, "tree k"
    assert close(g["tv"][b][ok], r.v[ok]) <= 0, "tree v"
    assert close(g["o"][b][ok], r.o[ok]) <= 0, "attention o"
    assert close(g["hp"][b][ok], r.hp[ok]) <= 0, "h'"
    assert close(g["vlog"][b][ok], r.zv[ok]) <= 0, "verification logits"
    am_bad = np.zeros(n1, dtype=bool)
    for n in range(n1):
        if r.am_margin[n] < NEAR:
            report["near_ties"] += 1
        if ok[n] and g["am"][b, n] != r.am[n]:
            if r.am_margin[n] < NEAR:
                excused.append(f"argmax node {n}")
                am_bad[n] = True
                continue
            raise AssertionError(f"argmax node {n}: {g['am'][b, n]} != {r.am[n]}")
    gm = int(g["n_acc"][b]) - 1
    g_path = [int(x) for x in g["path"][b, :gm + 1]]
    assert (g["path"][b, gm + 1:] == -1).all()
    assert list(g["out_tok"][b, :gm + 1]) == [int(g["tok"][b, n]) for n in g_path]
    assert (g["out_tok"][b, gm + 1:] == -1).all()
    np.testing.assert_array_equal(g["h_next"][b], g["hp"][b, g_path[-1]])   # h' of the last kept node
    if w.mode == "reject" and w.temperature > 0:
        # rejection sampling: the walk and the draw; the first choice that differs must be
        # within NEAR_P (probability units) of its boundary in the oracle
        o_path = [int(x) for x in r.path_nodes]
        same = g_path == o_path and int(g["root_next"][b]) == r.root_next
        if not same:
            i = 0
            while i < min(len(g_path), len(o_path)) and g_path[i] == o_path[i]:
                i += 1
            at = min(i, len(o_path)) - 1            # last common kept node: its choice differs
            u = o_path[at]
            touched = aff[u] or any(aff[c] for c in O.children(spec, u))
            if touched or r.rs_margins[at] < O.NEAR_P:
                excused.append(f"rejection walk at kept node {o_path[at]}")
            else:
                raise AssertionError(f"rejection walk {g_path} -> {g['root_next'][b]} != "
                                     f"{o_path} -> {r.root_next}")
        else:
            assert close(g["h_next"][b], r.h_next) <= 0, "h_next"
        if excused:
            raise Flagged(", ".join(excused))
        return
    # acceptance, node by node: the GPU's flags from its own statistics against the oracle's
    gacc, amb = gpu_accept_flags(g, b, spec, w)
    greedy = w.mode == "greedy" or w.temperature == 0
    acc_bad = np.zeros(n1, dtype=bool)
    for c in range(1, n1):
        p = spec.parent[c]
        if r.acc_margin[c] < NEAR:
            report["near_ties"] += 1
        if aff[c] or aff[p] or (greedy and am_bad[p]):
            acc_bad[c] = True                        # depends on an excused decision
            continue
        if gacc[c] != r.acc[c]:
            if r.acc_margin[c] < NEAR or amb[c]:
                excused.append(f"accept node {c}")
                acc_bad[c] = True
                continue
            raise AssertionError(f"accept flag of node {c}: gpu {gacc[c]} != oracle {r.acc[c]} "
                                 f"(margin {r.acc_margin[c]:.3g})")
    # the kept path is the longest accepted prefix of the GPU's own flags
    if not amb.any():
        _, _, m, nodes = O.longest_accepted(spec, gacc)
        assert m == gm and list(nodes) == g_path, "path is not the longest accepted prefix"
    if excused:
        assert explain_by_flips(spec, r, g_path, acc_bad), "path not explained by excused flips"
        raise Flagged(", ".join(excused))
    assert g_path == [int(x) for x in r.path_nodes], \
        f"accepted path {g_path} (m={gm}) != {list(r.path_nodes)} (m={r.m})"
    assert list(g["out_tok"][b, :gm + 1]) == list(r.out_tok)
    assert g["root_next"][b] == r.root_next or r.am_margin[g_path[-1]] < NEAR
    assert close(g["h_next"][b], r.h_next) <= 0, "h_next"


def record(case: str, compared: int, flagged: list):
    """Per-case counts of fully compared and flagged sequences, printed at the end of the
    pytest run."""
    from flag_report import RESULTS
    RESULTS[case] = (compared, flagged)
