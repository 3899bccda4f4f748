"""fp64 CPU oracle of one Medusa draft-and-verify decode step.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports, links or executes this file;
only the tests, the smoke check and the benchmark's CPU-baseline leg do.  It shares no
code with the CUDA path: both only read the seeded tensors of the `synthetic` package.

Plain, slow and meant to be checked by eye: numpy in float64, matrix-vector products as
the only library primitive, Python loops elsewhere.  Each function follows the step of
the method it names, in the order the pages give.  Sources:

  [MEDUSA]  "Medusa: Simple LLM Inference Acceleration Framework with Multiple Decoding
            Heads" (structured summary of arXiv 2401.10774), Section 3.
  [NOTES]   "Accelerating LLM Inference with Speculative Decoding: Notes on Medusa",
            sections 3 (Tree Attention) and 4 (Optimized Tree Construction).
  [READING] "MEDUSA 精读" (close reading), section 3 (draft tree, tree attention, verify)
            and section 6 (implementation checklist).

Readings where the pages are silent or disagree (each also listed in the design notes):
  R0  The backbone is one synthetic attention layer: x = E[tok]; q,k,v = Wq x, Wk x, Wv x
      per head; rotate-half RoPE with theta_i = base^(-2i/dh); softmax attention;
      h' = x + Wo o.  No norms, MLP or biases.  Cached prefix keys are post-RoPE.
  R1  Heads have no bias; the root (depth 0) is the LM head's single greedy token.
  R2  Top-s ranks by value descending, ties by lower token index.
  R3  Canonical packing: root first, then nodes by depth, then by rank path.
  R4  Each node attends to the whole prefix and to its own ancestors (itself included).
  R5  Greedy argmax takes the lowest index on ties; typical acceptance uses the strict
      ">" of [MEDUSA]'s criterion; at temperature 0 typical acceptance is greedy.
  R6  Best path = longest accepted prefix, ties to the lowest path index (paths are
      ordered by their leaf's packed index).  The next root is the greedy token at the
      last accepted node; the next hidden state is that node's h'.
  R7  Greedy tree construction adds, at each step, the frontier node with the largest
      path product of marginal accuracies ([NOTES] section 4 E[L] over all nodes);
      ties go to the lexicographically smaller rank path.
  R8  Rejection-sampling verification ([MEDUSA] §3.4, the speculative-decoding rule:
      accept a draft x with probability min(1, p(x)/q(x)), else draw from
      norm(max(0, p - q))).  The candidates are the heads' top-s tokens, i.e. drafts
      with a point-mass q = delta_x, so x is accepted with probability p(x) and a
      rejection removes x from p.  Walking from the root, the current node's children
      are tried in packed (rank) order against the remaining mass R: child x is accepted
      iff u < p(x) / R (u its own uniform), else R -= p(x); the first accepted child
      becomes the current node (fresh p, R = 1).  When no child is accepted (or the node
      has none) the next token is drawn from the remaining distribution at the current
      node by inverse CDF in token order (the smallest v whose cumulative remaining
      weight exceeds u_final times the remaining total); it is the next step's root.
      p = softmax(z / T); T = 0 is greedy.  Uniforms are inputs: uniforms[0] for the
      draw, uniforms[1 + (d - 1) * 16 + j] for the j-th child tried at depth d.
  R14 A backbone of n synthetic layers (the multi-layer form of R0 for a real backbone's
      per-layer calls): x_0 = E[tok]; layer l takes q, k, v from x_l with its own
      projections (RoPE at the node position), attends over its own prefix cache plus
      its own tree keys under the same mask, and x_{l+1} = x_l + Wo_l o_l; h' = x_n.
      Compaction appends the kept nodes' layer-l keys/values to layer l's cache.  With
      one layer this is R0.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

NEAR = 1e-3   # decisions whose fp64 margin is below this are flagged, not failed


# ============================================================ heads  [MEDUSA] §3.4
def silu(x):
    """SiLU(x) = x * sigmoid(x) = x / (1 + e^-x)."""
    return x / (1.0 + np.exp(-x))


def matvec(W, x, block=4096):
    """fp64 W @ x for a [rows][cols] numpy matrix stored as float32 or float64.

    float32 rows are converted to float64 a block at a time only to bound memory;
    every output is one plain dot product of a converted row with x.
    """
    W = np.asarray(W)
    if W.dtype == np.float64:
        return W @ x
    out = np.empty(W.shape[0], dtype=np.float64)
    for r in range(0, W.shape[0], block):
        out[r:r + block] = W[r:r + block].astype(np.float64) @ x
    return out


def oracle_weights(wts):
    """Harness conversion of the synthetic weights (torch, bf16 or fp32) to numpy.

    bf16 and fp32 values are exact in float64.  The K vocab projections W2 and the
    embedding stay float32 (exact as well) to bound memory; matvec widens them.
    """
    import torch
    out = {}
    for name, t in wts.items():
        keep32 = name in ("w2", "emb")
        out[name] = t.to(torch.float32 if keep32 else torch.float64).numpy()
    return out


def medusa_head(W1, W2, h):
    """Head k's logits: W2 (SiLU(W1 h) + h)  ([MEDUSA] §3.4 'MEDUSA Heads' equation).

    The softmax of the equation is left out: only the ranking of these logits is used
    downstream, and softmax is monotone.  Returns (u, logits), u = SiLU(W1 h) + h.
    """
    u = silu(matvec(W1, h)) + h
    return u, matvec(W2, u)


def lm_head(LM, h):
    """The original LM head's logits z0 = LM h (prediction for the next token)."""
    return matvec(LM, h)


def top_s(z, s):
    """The s most probable tokens: order by logit descending, then token index (R2).

    Returns (indices, values, margins): margins[r] is the smaller gap between the r-th
    value and its neighbours in the sorted order (including the (s+1)-th), i.e. how far
    rank r is from changing place.
    """
    order = sorted(range(len(z)), key=lambda v: (-z[v], v))
    vals = [z[v] for v in order[:s + 1]]
    margins = []
    for r in range(s):
        gaps = []
        if r > 0:
            gaps.append(vals[r - 1] - vals[r])
        if r + 1 < len(vals):
            gaps.append(vals[r] - vals[r + 1])
        margins.append(min(gaps) if gaps else math.inf)
    return np.array(order[:s], dtype=np.int64), np.array(vals[:s]), np.array(margins)


def argmax_lowest(z):
    """Greedy token: the largest logit, lowest index on ties (numpy's argmax returns the
    first occurrence of the maximum); also its top-2 margin."""
    z = np.asarray(z)
    best = int(np.argmax(z))
    rest = np.delete(z, best)
    second = rest.max() if rest.size else -math.inf
    return best, float(z[best] - second)


# ============================================================ tree  [MEDUSA] §3.4
@dataclass
class TreeSpec:
    """A packed candidate tree: node 0 is the root, parent[n] < n for n >= 1.

    paths[n] is node n's rank path (i_1, ..., i_depth); rank[n] = its last entry.
    """
    paths: list
    parent: list = field(default_factory=list)
    rank: list = field(default_factory=list)
    depth: list = field(default_factory=list)

    @property
    def N(self):
        return len(self.paths) - 1


def pack_tree(paths):
    """Canonical packing (R3): root, then nodes by depth, then by rank path."""
    paths = sorted(set(tuple(p) for p in paths if len(p) > 0), key=lambda p: (len(p), p))
    paths = [()] + paths
    index = {p: n for n, p in enumerate(paths)}
    parent = [-1] + [index[p[:-1]] for p in paths[1:]]
    rank = [0] + [p[-1] for p in paths[1:]]
    depth = [len(p) for p in paths]
    return TreeSpec(paths, parent, rank, depth)


def cartesian_tree(s):
    """Cartesian product of the per-head top-s_k ([MEDUSA] §3.4 Tree Attention, Step 2).

    Level k holds prod_{i<=k} s_i nodes, one per rank path (i_1..i_k), i_j < s_j.
    """
    paths = []
    level = [()]
    for sk in s:
        level = [p + (i,) for p in level for i in range(sk)]
        paths += level
    return pack_tree(paths)


def greedy_tree(a, s, N):
    """Optimized tree: greedy node addition under a node budget (R7).

    a[k][i] is head (k+1)'s marginal accuracy at rank i ([MEDUSA] §3.4 'Optimized Tree
    Construction', Steps 1-4; [NOTES] section 4).  A path's score is the product of its
    accuracies (independence assumption).  Starting from the root, repeatedly add the
    frontier node (a child of a chosen node, or of the root) with the largest score.
    """
    K = len(s)
    chosen = []
    frontier = {(i,): a[0][i] for i in range(s[0])}
    while len(chosen) < N and frontier:
        best = min(frontier, key=lambda p: (-frontier[p], p))
        score = frontier.pop(best)
        chosen.append(best)
        depth = len(best)
        if depth < K:
            for i in range(s[depth]):
                frontier[best + (i,)] = score * a[depth][i]
    return pack_tree(chosen)


def expected_accept_length(spec, a):
    """E[L] = sum over all tree nodes of the product of accuracies on the node's path
    ([NOTES] section 4, items 3-4)."""
    total = 0.0
    for p in spec.paths[1:]:
        prod = 1.0
        for k, i in enumerate(p):
            prod *= a[k][i]
        total += prod
    return total


def tree_tokens(spec, root, topk):
    """Token of each packed node: the root token, else topk[depth-1][rank]."""
    return np.array([root] + [int(topk[spec.depth[n] - 1][spec.rank[n]])
                              for n in range(1, spec.N + 1)], dtype=np.int64)


def ancestors(spec, n):
    """Packed indices on the root -> n path, root first, n last."""
    chain = []
    while n >= 0:
        chain.append(n)
        n = spec.parent[n]
    return chain[::-1]


def tree_mask(spec):
    """M[i][j] = 1 iff node j is an ancestor of node i or i itself
    ([MEDUSA] §3.4 Tree Attention, Step 3)."""
    n1 = spec.N + 1
    M = np.zeros((n1, n1), dtype=np.uint8)
    for i in range(n1):
        for j in ancestors(spec, i):
            M[i, j] = 1
    return M


def tree_positions(spec, L):
    """Position id of each node: prefix length + tree depth
    ([MEDUSA] §3.4 Tree Attention, Step 4; [READING] section 3)."""
    return np.array([L + spec.depth[n] for n in range(spec.N + 1)], dtype=np.int64)


def retrieve_paths(spec):
    """One root -> leaf path per leaf, leaves in packed order ([READING] section 6:
    the flatten / restore indices)."""
    has_child = set(spec.parent[1:])
    return [ancestors(spec, n) for n in range(spec.N + 1) if n not in has_child]


# ============================================================ synthetic layer (R0)
def rope(x, pos, base):
    """Rotate-half rotary embedding of one head vector x [dh] at position pos."""
    dh = len(x)
    half = dh // 2
    out = np.empty(dh, dtype=np.float64)
    for i in range(half):
        theta = base ** (-2.0 * i / dh)
        c, s = math.cos(pos * theta), math.sin(pos * theta)
        out[i] = x[i] * c - x[i + half] * s
        out[i + half] = x[i + half] * c + x[i] * s
    return out


def layer_qkv(lw, tok, pos, Hq, Hkv, dh, base):
    """x = E[tok]; per-head q, k (RoPE at pos) and v.  Shapes [Hq][dh], [Hkv][dh]."""
    x = np.asarray(lw["emb"][tok], dtype=np.float64)
    q = matvec(lw["wq"], x).reshape(Hq, dh)
    k = matvec(lw["wk"], x).reshape(Hkv, dh)
    v = matvec(lw["wv"], x).reshape(Hkv, dh)
    q = np.stack([rope(q[h], pos, base) for h in range(Hq)])
    k = np.stack([rope(k[h], pos, base) for h in range(Hkv)])
    return x, q, k, v


def attend(q, keys, vals):
    """Softmax attention of one query over a key list: softmax(keys q / sqrt(dh)) vals."""
    s = keys @ q / math.sqrt(len(q))
    s = s - s.max()
    p = np.exp(s)
    p = p / p.sum()
    return p @ vals


def tree_attention(q, kc, vc, kt, vt, M):
    """Attention of every packed node over the prefix plus the tree, under the tree mask
    ([MEDUSA] §3.4 Tree Attention, Steps 3 and 5).

    q [n1][Hq][dh] queries; kc, vc [L][Hkv][dh] prefix keys/values, visible to every
    node; kt, vt [n1][Hkv][dh] the nodes' own keys/values; M [n1][n1] the mask, node j
    visible to node i iff M[i][j] = 1.  Query head h reads key/value head
    h // (Hq / Hkv).  Returns o [n1][Hq][dh].
    """
    n1, Hq, dh = q.shape
    G = Hq // kc.shape[1]
    o = np.empty_like(q)
    for i in range(n1):
        for h in range(Hq):
            g = h // G
            s_pre = kc[:, g, :] @ q[i, h] / math.sqrt(dh)
            s_tree = np.where(M[i] == 1, kt[:, g, :] @ q[i, h] / math.sqrt(dh), -np.inf)
            s = np.concatenate([s_pre, s_tree])
            p = np.exp(s - s.max())
            p = p / p.sum()
            o[i, h] = p[:len(s_pre)] @ vc[:, g, :] + p[len(s_pre):] @ vt[:, g, :]
    return o


def layer_out(lw, x, o):
    """h' = x + Wo o (o: the heads' outputs concatenated)."""
    return x + matvec(lw["wo"], o.reshape(-1))


# ============================================================ acceptance  [MEDUSA] §3.4
def softmax_T(z, T):
    y = z / T
    y = y - y.max()
    p = np.exp(y)
    return p / p.sum()


def entropy(p):
    """H(p) = -sum p log p in nats."""
    nz = p[p > 0]
    return float(-(nz * np.log(nz)).sum())


def typical_accept(z, x, T, eps, delta):
    """Typical acceptance ([MEDUSA] §3.4 'Typical Acceptance Scheme'): accept x iff
    p(x) > min(eps, delta * exp(-H(p))), p the backbone's distribution at temperature T.
    Returns (accepted, margin) with margin = |log p(x) - log threshold|."""
    p = softmax_T(z, T)
    thr = min(eps, delta * math.exp(-entropy(p)))
    px = p[x]
    lp = math.log(px) if px > 0 else -math.inf
    return bool(px > thr), abs(lp - math.log(thr))


def accept_flags(spec, tok, zv, am, am_margin, accept):
    """Accept flag of every node ([MEDUSA] §3.4 'Typical Acceptance Scheme',
    'Whole-candidate and first-token handling'; [READING] section 4).

    The root (the LM head's greedy token) is always kept.  Candidate c is checked
    against the backbone's distribution at its parent p = parent[c]: greedy accepts iff
    tok[c] is p's greedy token; typical accepts iff p(tok[c]) > min(eps, delta e^-H).
    Typical at temperature 0 is greedy.  Returns (acc[n1], margin[n1]).
    """
    n1 = spec.N + 1
    T = accept.get("temperature", 0.0)
    greedy = accept["mode"] == "greedy" or T == 0.0
    acc = np.zeros(n1, dtype=np.int64)
    margin = np.full(n1, np.inf)
    acc[0] = 1
    for c in range(1, n1):
        p = spec.parent[c]
        if greedy:
            acc[c] = int(tok[c] == am[p])
            margin[c] = am_margin[p]
        else:
            ok, mar = typical_accept(zv[p], int(tok[c]), T, accept["eps"], accept["delta"])
            acc[c], margin[c] = int(ok), mar
    return acc, margin


NEAR_P = 1e-4   # rejection sampling: decisions within this (probability units) are flagged


def children(spec, u):
    """Packed indices of node u's children, in packed (rank) order."""
    return [c for c in range(1, spec.N + 1) if spec.parent[c] == u]


def inverse_cdf_draw(weights, u):
    """The smallest index v with sum(weights[:v+1]) > u * sum(weights) (R8), and the
    distance of that threshold to the nearest cumulative boundary, in units of the total.
    Zero weights are never drawn."""
    total = float(np.sum(weights))
    thr = u * total
    cum = 0.0
    last = -1
    for v, w in enumerate(weights):
        if w <= 0.0:
            continue
        last = v
        if cum + w > thr:
            return v, min(thr - cum, cum + w - thr) / total
        cum += w
    return last, 0.0


def rejection_walk(spec, tok, zv, T, uniforms):
    """Rejection-sampling verification of the candidate tree (R8).

    tok: [N+1] node tokens; zv: [N+1][V] verification logits; uniforms: [1 + 16 K].
    Returns (packed indices of the kept nodes root..last, the drawn next token, the
    decision margins in probability units: entry i is the smallest margin of the choice
    made at kept node i, i.e. its children's tries and, at the last node, the draw)."""
    path = [0]
    u = 0
    margins = []
    while True:
        p = softmax_T(zv[u], T)
        R = 1.0
        excluded = []
        nxt = None
        here = math.inf
        d = len(path)                                  # depth of the children tried
        for j, c in enumerate(children(spec, u)):
            x = int(tok[c])
            uu = float(uniforms[1 + (d - 1) * 16 + j])
            here = min(here, abs(uu * R - p[x]))
            if uu * R < p[x]:
                nxt = c
                break
            R -= p[x]
            excluded.append(x)
        if nxt is None:
            w = p.copy()
            w[excluded] = 0.0
            v, mar = inverse_cdf_draw(w, float(uniforms[0]))
            margins.append(min(here, mar))
            return np.array(path, dtype=np.int64), v, np.array(margins)
        margins.append(here)
        path.append(nxt)
        u = nxt


def longest_accepted(spec, acc):
    """The longest accepted prefix among all root -> leaf paths (R6).

    A path's length m counts its consecutive accepted nodes after the root.  Returns
    (m per path, best path index, m of the best path, packed indices of the kept nodes
    root..last).  Ties go to the lowest path index.
    """
    paths = retrieve_paths(spec)
    lens = np.zeros(len(paths), dtype=np.int64)
    for pi, path in enumerate(paths):
        m = 0
        while m + 1 < len(path) and acc[path[m + 1]]:
            m += 1
        lens[pi] = m
    best = int(np.argmax(lens))                    # first maximum = lowest path index
    m = int(lens[best])
    return lens, best, m, np.array(paths[best][:m + 1], dtype=np.int64)


# ============================================================ one decode step
@dataclass
class StepResult:
    z0: np.ndarray = None          # [V] LM-head logits at h_t
    u: np.ndarray = None           # [K][d] SiLU(W1 h) + h
    zk: np.ndarray = None          # [K][V] head logits
    topk: np.ndarray = None        # [K][s_max] token ids (-1 past s_k)
    topk_val: np.ndarray = None    # [K][s_max]
    topk_margin: np.ndarray = None
    root: int = 0
    root_margin: float = math.inf
    rs_margin: float = math.inf    # rejection sampling: smallest decision margin (R8)
    rs_margins: np.ndarray = None  # rejection sampling: margin of the choice at each kept node
    tok: np.ndarray = None         # [N+1]
    pos: np.ndarray = None         # [N+1]
    q: np.ndarray = None           # [N+1][Hq][dh]
    k: np.ndarray = None           # [N+1][Hkv][dh] tree keys (post-RoPE)
    v: np.ndarray = None           # [N+1][Hkv][dh]
    o: np.ndarray = None           # [N+1][Hq][dh] attention outputs
    hp: np.ndarray = None          # [N+1][d] h'
    zv: np.ndarray = None          # [N+1][V] verification logits
    am: np.ndarray = None          # [N+1] greedy token per node
    am_margin: np.ndarray = None
    acc: np.ndarray = None         # [N+1] accept flag per node (root: 1)
    acc_margin: np.ndarray = None  # [N+1] margin of the decision taken at each node
    path_len: np.ndarray = None    # [P] accepted nodes past the root per path
    best: int = 0
    m: int = 0                     # accepted candidates (n_acc = 1 + m)
    out_tok: np.ndarray = None     # [1+m]
    path_nodes: np.ndarray = None  # [1+m] packed indices of the kept nodes
    root_next: int = 0
    h_next: np.ndarray = None
    kv_new: tuple = None           # ([1+m][Hkv][dh], [1+m][Hkv][dh]) appended to the cache


def f64(t):
    """A weight or input tensor (torch or numpy, any float dtype) as float64 numpy."""
    try:
        import torch
        if isinstance(t, torch.Tensor):
            return t.to(torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(t, dtype=np.float64)


def heads_step(wts, h, s_max, s):
    """Steps (2)-(3) of [MEDUSA] §3.2's information flow for one sequence: the LM head
    and K Medusa heads on h, the root (greedy on z0) and per-head top-s_k."""
    r = StepResult()
    K = len(s)
    r.z0 = lm_head(wts["lm"], h)
    r.root, r.root_margin = argmax_lowest(r.z0)
    r.u = np.empty((K, len(h)))
    r.zk = np.empty((K, wts["lm"].shape[0]))
    r.topk = -np.ones((K, s_max), dtype=np.int64)
    r.topk_val = np.full((K, s_max), -np.inf)
    r.topk_margin = np.full((K, s_max), np.inf)
    for k in range(K):
        r.u[k], r.zk[k] = medusa_head(wts["w1"][k], wts["w2"][k], h)
        idx, val, mar = top_s(r.zk[k], s[k])
        r.topk[k, :s[k]], r.topk_val[k, :s[k]], r.topk_margin[k, :s[k]] = idx, val, mar
    return r


def medusa_step(wts, h, kc, vc, spec, dims, accept, root=None, s=None):
    """One decode step of one sequence, following [MEDUSA] §3.2's information flow.

    wts: weight tensors (see synthetic.weights); h: [d] last hidden state; kc, vc: the
    prefix's post-RoPE keys/values [L][Hkv][dh]; spec: packed TreeSpec; dims: dict with
    Hq, Hkv, dh, rope_base; accept: dict(mode, temperature, eps, delta); root: the
    carried-over first token, or None to take it from the LM head on h.
    """
    Hq, Hkv, dh, base = dims["Hq"], dims["Hkv"], dims["dh"], dims["rope_base"]
    h = f64(h)
    kc, vc = f64(kc), f64(vc)
    L = kc.shape[0]
    K = max(spec.depth)
    s = s or [max(p[k] for p in spec.paths if len(p) > k) + 1 for k in range(K)]
    s_max = max(s)

    # (2)-(3) heads, top-s, root
    r = heads_step(wts, h, s_max, s)
    if root is not None:
        r.root, r.root_margin = int(root), math.inf

    # (3) candidate tree: tokens and position ids
    n1 = spec.N + 1
    r.tok = tree_tokens(spec, r.root, r.topk)
    r.pos = tree_positions(spec, L)

    # (4) tree attention through the synthetic layer
    X = np.stack([np.asarray(wts["emb"][int(t)], dtype=np.float64) for t in r.tok])
    Q = (X @ np.asarray(wts["wq"], dtype=np.float64).T).reshape(n1, Hq, dh)
    Kt = (X @ np.asarray(wts["wk"], dtype=np.float64).T).reshape(n1, Hkv, dh)
    r.v = (X @ np.asarray(wts["wv"], dtype=np.float64).T).reshape(n1, Hkv, dh)
    r.q = np.stack([[rope(Q[n, h], r.pos[n], base) for h in range(Hq)]
                    for n in range(n1)])
    r.k = np.stack([[rope(Kt[n, h], r.pos[n], base) for h in range(Hkv)]
                    for n in range(n1)])
    r.o = tree_attention(r.q, kc, vc, r.k, r.v, tree_mask(spec))
    r.hp = np.stack([layer_out(wts, X[n], r.o[n]) for n in range(n1)])
    return _verify(r, wts, spec, accept)


def verify_only(wts, hp, tok, spec, accept):
    """Steps (5)-(6) alone, from given layer outputs hp [N+1][d] and node tokens tok
    [N+1]: the verification logits LM hp_n, acceptance, the kept path and the next root /
    hidden state ([MEDUSA] §3.4 Tree Attention Step 6 and Typical Acceptance Scheme)."""
    n1 = spec.N + 1
    r = StepResult()
    r.tok = np.asarray(tok, dtype=np.int64)
    r.hp = f64(hp)
    r.k = np.zeros((n1, 1))
    r.v = np.zeros((n1, 1))
    return _verify(r, wts, spec, accept)


def _verify(r, wts, spec, accept):
    """Steps (5)-(6) from the layer outputs r.hp: verification logits, acceptance, the
    kept path, the next root / hidden state, and the kept nodes' keys/values (r.k, r.v)."""
    n1 = spec.N + 1
    # verification logits ([MEDUSA] §3.4 Tree Attention, Step 6)
    r.zv = (np.asarray(wts["lm"], dtype=np.float64) @ r.hp.T).T   # z_n = LM h'_n
    r.am = np.empty(n1, dtype=np.int64)
    r.am_margin = np.empty(n1)
    for n in range(n1):
        r.am[n], r.am_margin[n] = argmax_lowest(r.zv[n])

    # (5) acceptance of each candidate, then the longest accepted prefix
    T = accept.get("temperature", 0.0)
    if accept["mode"] == "reject" and T > 0.0:
        # R8: rejection sampling walks the tree with the given uniforms
        r.path_nodes, r.root_next, r.rs_margins = rejection_walk(spec, r.tok, r.zv, T,
                                                                 accept["uniforms"])
        r.rs_margin = float(np.min(r.rs_margins))
        r.m = len(r.path_nodes) - 1
        r.acc = np.zeros(n1, dtype=np.int64)
        r.acc[r.path_nodes] = 1
        r.acc_margin = np.full(n1, np.inf)
        r.out_tok = r.tok[r.path_nodes]
        last = int(r.path_nodes[-1])
        r.h_next = r.hp[last].copy()
        r.kv_new = (r.k[r.path_nodes].copy(), r.v[r.path_nodes].copy())
        return r
    greedy_accept = dict(accept, mode="greedy") if accept["mode"] == "reject" else accept
    r.acc, r.acc_margin = accept_flags(spec, r.tok, r.zv, r.am, r.am_margin, greedy_accept)
    r.path_len, r.best, r.m, r.path_nodes = longest_accepted(spec, r.acc)
    r.out_tok = r.tok[r.path_nodes]
    last = int(r.path_nodes[-1])
    r.root_next = int(r.am[last])
    r.h_next = r.hp[last].copy()
    # (6) KV compaction: only the accepted path's keys/values join the cache
    r.kv_new = (r.k[r.path_nodes].copy(), r.v[r.path_nodes].copy())
    return r


# ============================================================ decoding loops
def sequential_greedy(wts, h, kc, vc, dims, n_tokens):
    """Plain greedy decoding, one token per forward pass, for the end-to-end pin.

    Token 0 is the LM head's greedy token on h; every later token is the greedy token
    of the layer output at the previous token.  Returns (tokens, final K, final V).
    """
    Hq, Hkv, dh, base = dims["Hq"], dims["Hkv"], dims["dh"], dims["rope_base"]
    G = Hq // Hkv
    K_, V_ = list(f64(kc)), list(f64(vc))
    tok, _ = argmax_lowest(lm_head(wts["lm"], f64(h)))
    out = []
    while len(out) < n_tokens:
        out.append(tok)
        pos = len(K_)
        x, q, k, v = layer_qkv(wts, tok, pos, Hq, Hkv, dh, base)
        K_.append(k)
        V_.append(v)
        Ka, Va = np.stack(K_), np.stack(V_)
        o = np.stack([attend(q[hq], Ka[:, hq // G], Va[:, hq // G]) for hq in range(Hq)])
        tok, _ = argmax_lowest(lm_head(wts["lm"], layer_out(wts, x, o)))
    return out, np.stack(K_), np.stack(V_)


def medusa_generate(wts, h, kc, vc, spec, dims, accept, n_steps):
    """Repeated decode steps carrying (h_next, root_next) and the compacted cache.

    Returns (tokens emitted, per-step results, final K, final V).
    """
    kc, vc = f64(kc), f64(vc)
    h = f64(h)
    root = None
    tokens, steps = [], []
    for _ in range(n_steps):
        r = medusa_step(wts, h, kc, vc, spec, dims, accept, root=root)
        steps.append(r)
        tokens += [int(t) for t in r.out_tok]
        kc = np.concatenate([kc, r.kv_new[0]])
        vc = np.concatenate([vc, r.kv_new[1]])
        h, root = r.h_next, r.root_next
    return tokens, steps, kc, vc


# ============================================================ multi-layer backbone (R14)
def medusa_step_layers(wts, layers, h, caches, spec, dims, accept, root=None, s=None):
    """One decode step of one sequence through an n-layer backbone (R14).

    layers: per layer a dict with wq, wk, wv, wo (layer 0's may be wts itself); caches:
    per layer (kc, vc) post-RoPE prefix keys/values [L][Hkv][dh] (the same L in every
    layer).  The result's k / v / q / o are layer 0's; layer_k / layer_v hold every
    layer's tree keys/values and kv_new_layers the kept nodes' per layer.
    """
    Hq, Hkv, dh, base = dims["Hq"], dims["Hkv"], dims["dh"], dims["rope_base"]
    h = f64(h)
    L = f64(caches[0][0]).shape[0]
    K = max(spec.depth)
    s = s or [max(p[k] for p in spec.paths if len(p) > k) + 1 for k in range(K)]
    r = heads_step(wts, h, max(s), s)
    if root is not None:
        r.root, r.root_margin = int(root), math.inf
    n1 = spec.N + 1
    r.tok = tree_tokens(spec, r.root, r.topk)
    r.pos = tree_positions(spec, L)
    M = tree_mask(spec)
    X = np.stack([np.asarray(wts["emb"][int(t)], dtype=np.float64) for t in r.tok])
    r.layer_k, r.layer_v = [], []
    for li, lw in enumerate(layers):
        kc, vc = f64(caches[li][0]), f64(caches[li][1])
        Q = (X @ f64(lw["wq"]).T).reshape(n1, Hq, dh)
        Kt = (X @ f64(lw["wk"]).T).reshape(n1, Hkv, dh)
        Vt = (X @ f64(lw["wv"]).T).reshape(n1, Hkv, dh)
        q = np.stack([[rope(Q[n, hh], r.pos[n], base) for hh in range(Hq)] for n in range(n1)])
        k = np.stack([[rope(Kt[n, hh], r.pos[n], base) for hh in range(Hkv)] for n in range(n1)])
        o = tree_attention(q, kc, vc, k, Vt, M)
        X = np.stack([layer_out(lw, X[n], o[n]) for n in range(n1)])
        r.layer_k.append(k)
        r.layer_v.append(Vt)
        if li == 0:
            r.q, r.k, r.v, r.o = q, k, Vt, o
    r.hp = X
    r = _verify(r, wts, spec, accept)
    r.kv_new_layers = [(k[r.path_nodes].copy(), v[r.path_nodes].copy())
                       for k, v in zip(r.layer_k, r.layer_v)]
    return r


def sequential_greedy_layers(wts, layers, h, caches, dims, n_tokens):
    """Plain greedy decoding through the n-layer backbone, one token per forward pass.
    Returns (tokens, final caches as a list of (K, V))."""
    Hq, Hkv, dh, base = dims["Hq"], dims["Hkv"], dims["dh"], dims["rope_base"]
    G = Hq // Hkv
    Ks = [list(f64(c[0])) for c in caches]
    Vs = [list(f64(c[1])) for c in caches]
    tok, _ = argmax_lowest(lm_head(wts["lm"], f64(h)))
    out = []
    while len(out) < n_tokens:
        out.append(tok)
        pos = len(Ks[0])
        x = np.asarray(wts["emb"][tok], dtype=np.float64)
        for li, lw in enumerate(layers):
            q = np.stack([rope(qh, pos, base) for qh in matvec(lw["wq"], x).reshape(Hq, dh)])
            k = np.stack([rope(kh, pos, base) for kh in matvec(lw["wk"], x).reshape(Hkv, dh)])
            v = matvec(lw["wv"], x).reshape(Hkv, dh)
            Ks[li].append(k)
            Vs[li].append(v)
            Ka, Va = np.stack(Ks[li]), np.stack(Vs[li])
            o = np.stack([attend(q[hq], Ka[:, hq // G], Va[:, hq // G]) for hq in range(Hq)])
            x = layer_out(lw, x, o)
        tok, _ = argmax_lowest(lm_head(wts["lm"], x))
    return out, [(np.stack(a), np.stack(b)) for a, b in zip(Ks, Vs)]


def medusa_generate_layers(wts, layers, h, caches, spec, dims, accept, n_steps):
    """Repeated n-layer decode steps carrying (h_next, root_next) and every layer's
    compacted cache.  Returns (tokens, per-step results, final caches)."""
    caches = [(f64(a), f64(b)) for a, b in caches]
    h = f64(h)
    root = None
    tokens, steps = [], []
    for _ in range(n_steps):
        r = medusa_step_layers(wts, layers, h, caches, spec, dims, accept, root=root)
        steps.append(r)
        tokens += [int(t) for t in r.out_tok]
        caches = [(np.concatenate([kc, kn]), np.concatenate([vc, vn]))
                  for (kc, vc), (kn, vn) in zip(caches, r.kv_new_layers)]
        h, root = r.h_next, r.root_next
    return tokens, steps, caches
