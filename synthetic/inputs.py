"""Seeded synthetic inputs shaped like the Medusa paper's Vicuna / Zephyr workloads.

This module holds no part of the method's arithmetic: only workload shapes, value
distributions and seeded random streams.  Both the fp64 oracle and the CUDA path read
their inputs from here; nothing else is shared between them.

The paper's evaluations (MT-Bench, AlpacaEval on Vicuna-7B/13B/33B and Zephyr-7B;
"MEDUSA: Simple LLM Inference Acceleration Framework with Multiple Decoding Heads",
Section 3 / Table 1) need trained weights and datasets.  These tensors stand in for
them with the same model shapes:

* weights ~ N(0, 1/fan_in) (embedding rows ~ N(0, 1)), last hidden state h_t ~ N(0, 1),
  KV prefix ~ N(0, 1) read as already-rotated keys;
* bf16 workloads store every tensor rounded once to bf16; h_t is handed over as the
  fp32 value of its bf16 rounding;
* each tensor has its own seeded stream ([seed, tag, index] -> numpy SeedSequence), so
  one sequence of a batch can be regenerated without the others.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import numpy as np
import torch

_TAGS = {"w1": 1, "w2": 2, "lm": 3, "emb": 4, "wq": 5, "wk": 6, "wv": 7, "wo": 8,
         "h": 9, "kc": 10, "vc": 11, "len": 12, "pages": 13, "perm": 14, "rho": 15,
         "uni": 16}


@dataclass(frozen=True)
class Workload:
    """One decode-step configuration (sizes follow the paper's model shapes)."""
    name: str
    B: int            # sequences in the batch
    d: int            # hidden size
    V: int            # vocabulary
    Hq: int           # query heads
    Hkv: int          # key/value heads (GQA when < Hq)
    dh: int           # head dim
    K: int            # Medusa heads
    dtype: str        # "f32" or "bf16": weights, embedding and KV cache
    lengths: tuple    # KV-prefix length per sequence
    tree: str         # "cartesian" or "greedy"
    s: tuple          # top-s_k kept per head k = 1..K
    N: int            # candidate nodes, root excluded
    mode: str = "greedy"          # "greedy" or "typical"
    temperature: float = 0.0
    eps: float = 0.09
    delta: float = 0.3
    page_size: int = 0            # 0: contiguous cache, else tokens per page
    seed: int = 0
    rope_base: float = 10000.0
    reserve: int = 128            # free KV slots kept beyond the longest prefix

    @property
    def capacity(self) -> int:
        """KV slots per sequence (multiple of 16 so it splits into whole pages)."""
        c = max(self.lengths) + self.reserve
        return (c + 15) // 16 * 16

    @property
    def pages_per_seq(self) -> int:
        return self.capacity // self.page_size if self.page_size else 0

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


def _lengths_uniform(seed: int, B: int, lo: int, hi: int) -> tuple:
    rng = np.random.default_rng(np.random.SeedSequence([seed, _TAGS["len"]]))
    return tuple(int(x) for x in rng.integers(lo, hi + 1, size=B))


WORKLOADS = {
    # tiny single step: fp32, top-(3,2,2) Cartesian tree = 21 nodes + root, greedy
    "tiny": Workload("tiny", B=1, d=128, V=512, Hq=4, Hkv=4, dh=32, K=3, dtype="f32",
                     lengths=(64,), tree="cartesian", s=(3, 2, 2), N=21),
    # Vicuna-7B-shaped step, greedy acceptance, 64-node sparse tree from top-10 per head
    "vicuna7b": Workload("vicuna7b", B=1, d=4096, V=32000, Hq=32, Hkv=32, dh=128, K=5,
                         dtype="bf16", lengths=(1024,), tree="greedy", s=(10,) * 5, N=64),
    # same with typical acceptance (eps=0.09, delta=0.3, T=0.7)
    "vicuna7b_typical": Workload("vicuna7b_typical", B=1, d=4096, V=32000, Hq=32, Hkv=32,
                                 dh=128, K=5, dtype="bf16", lengths=(1024,), tree="greedy",
                                 s=(10,) * 5, N=64, mode="typical", temperature=0.7),
    # Vicuna-13B-shaped, batch 8, prefix lengths uniform in [2048, 4096], typical T=0.7
    "vicuna13b": Workload("vicuna13b", B=8, d=5120, V=32000, Hq=40, Hkv=40, dh=128, K=5,
                          dtype="bf16", lengths=_lengths_uniform(0, 8, 2048, 4096),
                          tree="greedy", s=(10,) * 5, N=64, mode="typical",
                          temperature=0.7),
    # Zephyr-7B-shaped with GQA 32/8, batch 16, prefix 8192, paged cache of 16-token pages
    "zephyr7b": Workload("zephyr7b", B=16, d=4096, V=32000, Hq=32, Hkv=8, dh=128, K=4,
                         dtype="bf16", lengths=(8192,) * 16, tree="greedy", s=(10,) * 4,
                         N=42, page_size=16),
}


def vicuna33b(B: int, L: int, N: int) -> Workload:
    """One point of the Vicuna-33B-shaped sweep (B x prefix x tree size), greedy."""
    return Workload(f"vicuna33b_b{B}_l{L}_n{N}", B=B, d=6656, V=32000, Hq=52, Hkv=52,
                    dh=128, K=5, dtype="bf16", lengths=(L,) * B, tree="greedy",
                    s=(10,) * 5, N=N)


def workload(name: str, **overrides) -> Workload:
    w = WORKLOADS[name]
    return replace(w, **overrides) if overrides else w


# --------------------------------------------------------------------------- streams
def _rng(w: Workload, tag: str, index: int = 0) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([w.seed, _TAGS[tag], index]))


def _normal(w: Workload, tag: str, shape, std: float, index: int = 0) -> torch.Tensor:
    """N(0, std^2) fp32 values, rounded once to the workload's dtype."""
    a = _rng(w, tag, index).standard_normal(int(np.prod(shape)), dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return torch.from_numpy(a.reshape(shape)).to(w.torch_dtype)


def weights(w: Workload) -> dict:
    """Head, LM-head and one-layer backbone weights, stored [out][in] row-major."""
    d, V, K = w.d, w.V, w.K
    qd, kd = w.Hq * w.dh, w.Hkv * w.dh
    sd = 1.0 / math.sqrt(d)
    w1 = torch.empty((K, d, d), dtype=w.torch_dtype)
    w2 = torch.empty((K, V, d), dtype=w.torch_dtype)
    for k in range(K):                      # one stream per head keeps peak memory low
        w1[k] = _normal(w, "w1", (d, d), sd, k)
        w2[k] = _normal(w, "w2", (V, d), sd, k)
    return {
        "w1": w1, "w2": w2,
        "lm": _normal(w, "lm", (V, d), sd),
        "emb": _normal(w, "emb", (V, d), 1.0),
        "wq": _normal(w, "wq", (qd, d), sd),
        "wk": _normal(w, "wk", (kd, d), sd),
        "wv": _normal(w, "wv", (kd, d), sd),
        "wo": _normal(w, "wo", (d, qd), 1.0 / math.sqrt(qd)),
    }


def layer_weights(w: Workload, layer: int, planted: bool = False) -> dict:
    """Projections of backbone layer `layer` (0: the same tensors as `weights`), stored
    [out][in]: wq, wk, wv, wo.  Layers past 0 draw from their own streams; `planted`
    scales Wo by 0.1 as planted_weights does, so the residual stream stays dominant."""
    d, qd, kd = w.d, w.Hq * w.dh, w.Hkv * w.dh
    sd = 1.0 / math.sqrt(d)
    lw = {
        "wq": _normal(w, "wq", (qd, d), sd, layer),
        "wk": _normal(w, "wk", (kd, d), sd, layer),
        "wv": _normal(w, "wv", (kd, d), sd, layer),
        "wo": _normal(w, "wo", (d, qd), 1.0 / math.sqrt(qd), layer),
    }
    if planted:
        lw["wo"] = (lw["wo"].to(torch.float32) * 0.1).to(w.torch_dtype)
    return lw


def hidden(w: Workload) -> torch.Tensor:
    """Last hidden state h_t [B][d] as fp32 holding dtype-rounded N(0,1) values."""
    return _normal(w, "h", (w.B, w.d), 1.0).to(torch.float32)


def uniforms(w: Workload, step: int = 0) -> torch.Tensor:
    """Uniform draws in [0, 1) for rejection-sampling verification, [B][1 + 16 K] float32:
    [b][0] for the final draw, [b][1 + 16 (d - 1) + j] for the j-th child tried at depth d.
    One seeded stream per step."""
    a = _rng(w, "uni", step).random((w.B, 1 + 16 * w.K), dtype=np.float32)
    return torch.from_numpy(a)


def kv_prefix(w: Workload, b: int, layer: int = 0):
    """Post-RoPE prefix keys and values of sequence b in backbone layer `layer`: two
    [L_b][Hkv][dh] tensors."""
    shape = (w.lengths[b], w.Hkv, w.dh)
    i = b + 100000 * layer
    return _normal(w, "kc", shape, 1.0, i), _normal(w, "vc", shape, 1.0, i)


def page_table(w: Workload) -> torch.Tensor:
    """[B][pages_per_seq] int32 physical page ids: one seeded permutation of the pool."""
    P = w.pages_per_seq
    perm = _rng(w, "pages").permutation(w.B * P).astype(np.int32)
    return torch.from_numpy(perm.reshape(w.B, P))


def kv_cache(w: Workload, layer: int = 0):
    """Device-layout KV cache of backbone layer `layer` holding every sequence's prefix.

    Contiguous: K, V each [B][capacity][Hkv][dh].  Paged (page_size > 0): K, V each
    [B*pages_per_seq][page_size][Hkv][dh] plus the page table; logical slot t of
    sequence b lives in page page_table[b][t // page_size] at row t % page_size.
    Slots past the prefix hold zeros.
    """
    cap, Hkv, dh = w.capacity, w.Hkv, w.dh
    kc = torch.zeros((w.B, cap, Hkv, dh), dtype=w.torch_dtype)
    vc = torch.zeros((w.B, cap, Hkv, dh), dtype=w.torch_dtype)
    for b in range(w.B):
        k, v = kv_prefix(w, b, layer)
        kc[b, :w.lengths[b]] = k
        vc[b, :w.lengths[b]] = v
    if not w.page_size:
        return kc, vc, None
    ps, P = w.page_size, w.pages_per_seq
    pt = page_table(w)
    kp = torch.empty((w.B * P, ps, Hkv, dh), dtype=w.torch_dtype)
    vp = torch.empty_like(kp)
    for b in range(w.B):
        kp[pt[b].long()] = kc[b].reshape(P, ps, Hkv, dh)
        vp[pt[b].long()] = vc[b].reshape(P, ps, Hkv, dh)
    return kp, vp, pt


def kv_cache_device(w: Workload, host_seqs, device):
    """kv_cache built on `device` for caches too large to draw on the host in a test:
    the sequences in host_seqs get their prefixes from the host streams (the values
    kv_prefix gives the oracle); every other sequence's prefix is N(0, 1) drawn on the
    device from a generator seeded with the workload's seed.  Contiguous layout only."""
    if w.page_size:
        raise ValueError("kv_cache_device: contiguous caches only")
    cap, Hkv, dh = w.capacity, w.Hkv, w.dh
    kc = torch.zeros((w.B, cap, Hkv, dh), dtype=w.torch_dtype, device=device)
    vc = torch.zeros_like(kc)
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed * 1000003 + _TAGS["kc"])
    for b in range(w.B):
        L = w.lengths[b]
        if b in host_seqs:
            k, v = kv_prefix(w, b)
            kc[b, :L] = k.to(device)
            vc[b, :L] = v.to(device)
        else:
            for t in (kc, vc):
                t[b, :L] = torch.randn((L, Hkv, dh), generator=gen, device=device,
                                       dtype=torch.float32).to(w.torch_dtype)
    return kc, vc, None


def score_table(K: int, smax: int) -> np.ndarray:
    """Fixed node-score table a_k^(i) (marginal top-i accuracy of head k), [K][smax].

    Geometric marginals a_k^(i) = t_k (1 - t_k)^(i-1) with head accuracies t decreasing
    with k, the shape of the calibrated accuracies the paper describes for its
    optimized tree (Section 2.3.3).  The values are fixed, so the seed is not used.
    """
    t = [0.72, 0.55, 0.45, 0.38, 0.33, 0.29, 0.26, 0.24][:K]
    a = np.empty((K, smax), dtype=np.float64)
    for k in range(K):
        for i in range(smax):
            a[k, i] = t[k] * (1.0 - t[k]) ** i
    return a


def head_init_weights(wts: dict) -> dict:
    """The paper's head initialisation: W1 = 0 and every W2 equal to the LM head."""
    out = dict(wts)
    out["w1"] = torch.zeros_like(wts["w1"])
    out["w2"] = wts["lm"].unsqueeze(0).expand_as(wts["w2"]).contiguous()
    return out


def planted_weights(w: Workload, p_right: float = 0.7) -> dict:
    """Weights of a 'planted' model whose heads are often right, for long accepted paths.

    Embedding rows are random (near-orthogonal); token t is followed by pi(t) for a
    seeded permutation pi: LM row v = E[pi^-1(v)] / sqrt(d).  Head k's W2 row v is
    E[sigma_k^-1(v)] / sqrt(d) with sigma_k = rho_k o pi^(k+1), where rho_k fixes a
    p_right share of the tokens and permutes the rest, so head k's top-1 equals the
    true token k+1 steps ahead about p_right of the time.  W1 = 0; Wo is scaled by 0.1
    so the residual stream keeps the current token's embedding dominant.
    """
    wts = weights(w)
    d, V = w.d, w.V
    emb = wts["emb"].to(torch.float32)
    rng = _rng(w, "perm")
    pi = rng.permutation(V)

    def inv(p):
        q = np.empty_like(p)
        q[p] = np.arange(len(p))
        return q

    def rows_for(sigma):  # row v of the projection = E[sigma^-1(v)] / sqrt(d)
        return (emb[torch.from_numpy(inv(sigma))] / math.sqrt(d)).to(w.torch_dtype)

    wts["lm"] = rows_for(pi)
    w2 = torch.empty_like(wts["w2"])
    for k in range(w.K):
        target = _pow(pi, k + 2)        # head index k (0-based) looks k+2 tokens ahead
        r = _rng(w, "rho", k)
        moved = np.flatnonzero(r.random(V) >= p_right)
        rho = np.arange(V)
        rho[moved] = moved[r.permutation(len(moved))]
        w2[k] = rows_for(rho[target])
    wts["w2"] = w2
    wts["w1"] = torch.zeros_like(wts["w1"])
    wts["wo"] = (wts["wo"].to(torch.float32) * 0.1).to(w.torch_dtype)
    return wts


def _pow(p: np.ndarray, n: int) -> np.ndarray:
    out = np.arange(len(p))
    for _ in range(n):
        out = p[out]
    return out
