"""Failure detection on the GPU without a fault: a bounded wait inside a tensor-core
kernel is made to run out (it waits on a barrier that nothing arrives on), and the
library must report MEDUSA_FLAG_TIMEOUT through the status word, return, and leave the
plan and the CUDA context usable: the next step on the same plan matches the oracle."""
import time

import numpy as np
import pytest
import torch

import oracle as O
import synthetic as S
from medusa_head_speculative_gb300 import binding as Bnd

from harness import Flagged, compare_sequence, oracle_step, run_stages, run_step, setup

pytestmark = pytest.mark.gpu


def _mid(**kw):
    base = dict(name="mid", B=3, d=256, V=1000, Hq=8, Hkv=2, dh=64, K=4, dtype="bf16",
                lengths=(37, 100, 257), tree="greedy", s=(10, 10, 10, 10), N=30)
    base.update(kw)
    return S.Workload(**base)


@pytest.mark.parametrize("w", [_mid(), _mid(B=6, lengths=(40,) * 6, N=60, V=4000)],
                         ids=["narrow_gemm", "wide_gemm"])
def test_expired_wait_sets_timeout_and_the_plan_stays_usable(w):
    dev = setup(w)
    clean = run_step(dev, len_out=torch.empty_like(dev.length))
    assert dev.plan.status() == 0
    dev.plan.expire_wait_once(2_000_000)                 # 2 ms, then the expired-wait path
    t0 = time.perf_counter()
    run_step(dev, len_out=torch.empty_like(dev.length))  # returns (outputs meaningless)
    elapsed = time.perf_counter() - t0
    assert dev.plan.status() & Bnd.FLAG_TIMEOUT
    assert elapsed < 30.0
    assert dev.plan.status() == 0                       # reading cleared the word
    # the one-shot setting is gone: the same plan steps normally again ...
    again = run_step(dev, len_out=torch.empty_like(dev.length))
    assert dev.plan.status() == 0
    for k in ("out_tok", "n_acc", "path"):
        np.testing.assert_array_equal(again[k], clean[k])
    np.testing.assert_array_equal(again["h_next"].cpu().numpy(), clean["h_next"].cpu().numpy())
    # ... and its stages still match the oracle
    g = run_stages(dev)
    ow = O.oracle_weights(dev.cpu["wts"])
    compared = 0
    for b in range(w.B):
        try:
            compare_sequence(g, oracle_step(dev, b, ow), b, dev.spec, w, {})
            compared += 1
        except Flagged:
            pass
    assert compared >= w.B - 1


def test_expire_wait_argument_checks():
    dev = setup(_mid())
    with pytest.raises(Bnd.MedusaError):
        dev.plan.expire_wait_once(0)
    f32 = setup(_mid(dtype="f32"))
    with pytest.raises(Bnd.MedusaError) as e:
        f32.plan.expire_wait_once(1000)
    assert e.value.code == Bnd.MEDUSA_ERR_UNSUPPORTED
