"""The multi-layer backbone (medusa_step_layers) against the oracle's n-layer step (R14):
accepted tokens, path, next root and hidden state, and every layer's compacted cache; one
layer equals medusa_step bit for bit; on the planted tiny model a multi-step loop through
several layers emits the plain greedy continuation."""
import numpy as np
import pytest
import torch

import oracle as O
import synthetic as S
from medusa_head_speculative_gb300 import binding as Bnd

from harness import NEAR, accept_of, close, oracle_accept, run_step, setup

pytestmark = pytest.mark.gpu


def _mid(**kw):
    base = dict(name="mid", B=3, d=256, V=1000, Hq=8, Hkv=2, dh=64, K=4, dtype="bf16",
                lengths=(37, 100, 257), tree="greedy", s=(10, 10, 10, 10), N=30)
    base.update(kw)
    return S.Workload(**base)


def _layers(dev, n_layers, planted=False):
    """Device layers: layer 0 = the setup's projections and cache, then fresh ones."""
    w = dev.w
    layers = [dict(wq=dev.wts["wq"], wk=dev.wts["wk"], wv=dev.wts["wv"], wo=dev.wts["wo"],
                   k=dev.kc, v=dev.vc)]
    cpu = [dev.cpu["wts"]]
    for l in range(1, n_layers):
        lw = S.layer_weights(w, l, planted=planted)
        kc, vc, _ = S.kv_cache(w, l)
        layers.append(dict(**{k: t.cuda() for k, t in lw.items()}, k=kc.cuda(), v=vc.cuda()))
        cpu.append(lw)
    return layers, cpu


def _step_layers(dev, layers, root_in=None):
    w, p = dev.w, dev.plan
    i32 = dict(dtype=torch.int32, device="cuda")
    out_tok = torch.empty(w.B, w.K + 1, **i32)
    n_acc = torch.empty(w.B, **i32)
    path = torch.empty(w.B, w.K + 1, **i32)
    h_next = torch.empty(w.B, w.d, dtype=torch.float32, device="cuda")
    root_next = torch.empty(w.B, **i32)
    ws = torch.empty(p.workspace_size_layers(len(layers)), dtype=torch.uint8, device="cuda")
    kv = Bnd.kv_struct(None, None, dev.length, dev.length, dev.pt)
    outs = Bnd.outputs_struct(out_tok, n_acc, path, h_next, root_next)
    Bnd.step_layers(p, dev.h, root_in, dev.wstruct, Bnd.layers_array(layers), kv,
                    Bnd.accept_struct(**accept_of(w, dev)), outs, ws)
    torch.cuda.synchronize()
    assert p.status() == 0
    return dict(out_tok=out_tok.cpu().numpy(), n_acc=n_acc.cpu().numpy(), path=path.cpu().numpy(),
                h_next=h_next, root_next=root_next)


def _cache_rows(w, kc, pt, b, t0, n):
    """Rows t0 .. t0+n-1 of sequence b's cache (contiguous or paged) as fp64 numpy."""
    rows = []
    for t in range(t0, t0 + n):
        if pt is None:
            rows.append(kc[b, t])
        else:
            rows.append(kc[int(pt[b, t // w.page_size]), t % w.page_size])
    return torch.stack(rows).double().cpu().numpy()


def _flagged(r, w, root_given):
    """True when a decision the outputs depend on is a near tie in the oracle: the root,
    a used top-s rank, a node's acceptance, or the greedy token at the last kept node."""
    if not root_given and r.root_margin < NEAR:
        return True
    if np.min(r.topk_margin[np.isfinite(r.topk_margin)], initial=np.inf) < NEAR:
        return True
    if np.min(r.acc_margin) < NEAR or r.am_margin[int(r.path_nodes[-1])] < NEAR:
        return True
    return False


@pytest.mark.parametrize("w,n_layers", [
    (_mid(), 3),
    (_mid(mode="typical", temperature=0.7, page_size=16), 2),
    (S.workload("tiny"), 3),
    (S.Workload(name="tiny18", B=2, d=64, V=256, Hq=2, Hkv=2, dh=32, K=3, dtype="f32",
                lengths=(20, 33), tree="cartesian", s=(3, 2, 2), N=21), 18),
], ids=["mid_bf16_3", "mid_typical_paged_2", "tiny_f32_3", "tiny_f32_18"])
def test_layers_step_matches_oracle(w, n_layers):
    dev = setup(w)
    lengths = list(w.lengths)
    layers, cpu = _layers(dev, n_layers)
    g = _step_layers(dev, layers)
    ow = O.oracle_weights(dev.cpu["wts"])
    olayers = [O.oracle_weights(c) for c in cpu]
    dims = {"Hq": w.Hq, "Hkv": w.Hkv, "dh": w.dh, "rope_base": w.rope_base}
    new_len = dev.length.cpu().numpy()
    compared = 0
    for b in range(w.B):
        caches = [S.kv_prefix(w, b, l) for l in range(n_layers)]
        r = O.medusa_step_layers(ow, olayers, dev.cpu["h"][b], caches, dev.spec, dims,
                                 oracle_accept(w, b), s=list(w.s))
        if _flagged(r, w, False):
            continue
        n = r.m + 1
        assert g["n_acc"][b] == n
        assert list(g["out_tok"][b, :n]) == [int(t) for t in r.out_tok]
        assert list(g["path"][b, :n]) == [int(t) for t in r.path_nodes]
        assert int(g["root_next"][b]) == r.root_next
        assert close(g["h_next"][b].cpu().numpy(), r.h_next) <= 0, "h_next"
        assert new_len[b] == lengths[b] + n
        for l in range(n_layers):
            kn, vn = r.kv_new_layers[l]
            kg = _cache_rows(w, layers[l]["k"], dev.pt, b, lengths[b], n).reshape(kn.shape)
            vg = _cache_rows(w, layers[l]["v"], dev.pt, b, lengths[b], n).reshape(vn.shape)
            assert close(kg, kn) <= 0, f"layer {l} keys"
            assert close(vg, vn) <= 0, f"layer {l} values"
        compared += 1
    assert compared >= 1


def test_one_layer_equals_medusa_step():
    w = _mid()
    a = setup(w)
    ra = run_step(a)
    b = setup(w)
    layers, _ = _layers(b, 1)
    rb = _step_layers(b, layers)
    for k in ("out_tok", "n_acc", "path"):
        np.testing.assert_array_equal(ra[k], rb[k])
    np.testing.assert_array_equal(ra["h_next"].cpu().numpy(), rb["h_next"].cpu().numpy())
    np.testing.assert_array_equal(ra["root_next"].cpu().numpy(), rb["root_next"].cpu().numpy())
    np.testing.assert_array_equal(a.kc.float().cpu().numpy(), b.kc.float().cpu().numpy())
    np.testing.assert_array_equal(a.length.cpu().numpy(), b.length.cpu().numpy())


def test_planted_two_layer_loop_emits_sequential_greedy():
    """Medusa decoding of the planted tiny model through two layers, carrying root and h
    between medusa_step_layers calls, emits the plain greedy continuation."""
    w = S.workload("tiny")
    wts = S.planted_weights(w)
    h0 = wts["emb"][7].float().unsqueeze(0).clone()
    dev = setup(w, wts_cpu=wts, h_cpu=h0)
    layers, cpu = _layers(dev, 2, planted=True)
    toks, root, steps = [], None, 5
    for _ in range(steps):
        g = _step_layers(dev, layers, root_in=root)
        n = int(g["n_acc"][0])
        toks += [int(t) for t in g["out_tok"][0, :n]]
        dev.h = g["h_next"].clone()
        root = g["root_next"].clone()
    ow = O.oracle_weights(wts)
    olayers = [O.oracle_weights(c) for c in cpu]
    dims = {"Hq": w.Hq, "Hkv": w.Hkv, "dh": w.dh, "rope_base": w.rope_base}
    caches = [S.kv_prefix(w, 0, l) for l in range(2)]
    ref, _ = O.sequential_greedy_layers(ow, olayers, h0[0], caches, dims, len(toks))
    assert toks == ref
    assert len(toks) > steps                      # some step kept candidates past the root
