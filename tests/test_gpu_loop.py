"""The steady-state decode loop (medusa_loop_*): one medusa_step with its state carried in
place, captured as a CUDA graph and replayed, must equal the same steps called one by one
(bit for bit), and on the planted tiny model emit the oracle's Medusa / greedy tokens."""
import numpy as np
import pytest
import torch

import oracle as O
import synthetic as S
from medusa_head_speculative_gb300 import binding as Bnd

from harness import accept_of, run_step, setup

pytestmark = pytest.mark.gpu


def _mid(**kw):
    base = dict(name="mid", B=3, d=256, V=1000, Hq=8, Hkv=2, dh=64, K=4, dtype="bf16",
                lengths=(37, 100, 257), tree="greedy", s=(10, 10, 10, 10), N=30)
    base.update(kw)
    return S.Workload(**base)


def _loop(dev, root, steps):
    w = dev.w
    tokens = torch.full((steps, w.B, w.K + 1), -7, dtype=torch.int32, device="cuda")
    n_acc = torch.full((steps, w.B), -7, dtype=torch.int32, device="cuda")
    kv = Bnd.kv_struct(dev.kc, dev.vc, dev.length, dev.length, dev.pt)
    loop = Bnd.Loop(dev.plan, dev.wstruct, kv, Bnd.accept_struct(**accept_of(w)), dev.h, root,
                    tokens, n_acc, dev.ws)
    return loop, tokens, n_acc


@pytest.mark.parametrize("w", [_mid(), _mid(mode="typical", temperature=0.7, page_size=16),
                               S.workload("tiny")], ids=["mid_greedy", "mid_typical_paged", "tiny"])
def test_loop_equals_chained_steps(w):
    steps = 6
    # reference: the same steps through medusa_step, state carried by the caller
    ref = setup(w)
    s = run_step(ref)                                   # first step: root from the LM head
    ref.h, root = s["h_next"].clone(), s["root_next"].clone()
    toks, naccs = [], []
    for _ in range(steps):
        s = run_step(ref, root_in=root)
        ref.h, root = s["h_next"].clone(), s["root_next"].clone()
        toks.append(s["out_tok"])
        naccs.append(s["n_acc"])
    # the loop, from the same first step
    dev = setup(w)
    s = run_step(dev)
    dev.h = s["h_next"].clone()
    root_l = s["root_next"].clone()
    loop, tokens, n_acc = _loop(dev, root_l, steps)
    loop.run(steps)
    assert loop.steps() == steps
    assert dev.plan.status() == 0
    np.testing.assert_array_equal(tokens.cpu().numpy(), np.stack(toks))
    np.testing.assert_array_equal(n_acc.cpu().numpy(), np.stack(naccs))
    np.testing.assert_array_equal(dev.h.cpu().numpy(), ref.h.cpu().numpy())
    np.testing.assert_array_equal(root_l.cpu().numpy(), root.cpu().numpy())
    np.testing.assert_array_equal(dev.length.cpu().numpy(), ref.length.cpu().numpy())
    np.testing.assert_array_equal(dev.kc.float().cpu().numpy(), ref.kc.float().cpu().numpy())
    loop.close()


def test_loop_ring_wraps_and_keeps_counting():
    w = _mid()
    dev = setup(w)
    s = run_step(dev)
    dev.h = s["h_next"].clone()
    root = s["root_next"].clone()
    loop, tokens, n_acc = _loop(dev, root, 4)
    loop.run(3)
    loop.run(3)                                         # 6 steps into a ring of 4
    assert loop.steps() == 6
    assert (n_acc.cpu().numpy() >= 1).all()


def test_loop_on_planted_tiny_model_emits_the_oracle_tokens():
    """Medusa decoding of the planted tiny model through the loop = the oracle's Medusa loop
    = plain sequential greedy decoding."""
    w = S.workload("tiny")
    wts = S.planted_weights(w)
    h0 = wts["emb"][7].float().unsqueeze(0).clone()
    dev = setup(w, wts_cpu=wts, h_cpu=h0)
    ow = O.oracle_weights(wts)
    dims = {"Hq": w.Hq, "Hkv": w.Hkv, "dh": w.dh, "rope_base": w.rope_base}
    k0, v0 = S.kv_prefix(w, 0)
    steps = 8
    toks_o, steps_o, _, _ = O.medusa_generate(ow, h0[0], k0, v0, dev.spec, dims, {"mode": "greedy"},
                                              steps)
    s = run_step(dev)
    n = int(s["n_acc"][0])
    toks_g = list(s["out_tok"][0, :n])
    dev.h = s["h_next"].clone()
    root = s["root_next"].clone()
    loop, tokens, n_acc = _loop(dev, root, steps - 1)
    loop.run(steps - 1)
    t, a = tokens.cpu().numpy(), n_acc.cpu().numpy()
    for i in range(steps - 1):
        toks_g += list(t[i, 0, :a[i, 0]])
    assert toks_g == toks_o
    assert max(s_.m for s_ in steps_o) >= 2              # paths longer than the root alone
    loop.close()
