"""The workspace-free heads entry point (medusa_heads_noalloc).

It exists for callers that cannot hand the library freshly allocated device memory
while decoding: engines that plan all device memory before serving starts, plug-ins
confined to a host framework's memory pool, and code that may run during CUDA graph
capture.  Its scratch is one fixed device array owned by the library.

This file is collected last on purpose, so a run that stops at the first failure has
already run every other test.  It must pass both alone in a fresh process and after the
other tests.
"""
import numpy as np
import pytest
import torch

import synthetic as S
from medusa_head_speculative_gb300 import binding as Bnd

from harness import ATOL, RTOL, close, setup

pytestmark = pytest.mark.gpu


def _mid():
    return S.Workload("noalloc_mid", B=3, d=256, V=1000, Hq=8, Hkv=2, dh=64, K=4, dtype="bf16",
                      lengths=(37, 100, 257), tree="greedy", s=(10, 10, 10, 10), N=30)


@pytest.mark.parametrize("w", [S.workload("tiny"), _mid(), S.workload("vicuna7b")],
                         ids=["tiny", "mid", "vicuna7b"])
def test_noalloc_heads_matches_workspace_heads(w):
    dev = setup(w)
    p = dev.plan
    B, K = w.B, w.K
    i32 = dict(dtype=torch.int32, device="cuda")
    logits = torch.empty(B, K + 1, w.V, dtype=torch.float32, device="cuda")
    ref_tok, ref_val = torch.empty(B, K, 16, **i32), torch.empty(B, K, 16, device="cuda")
    ref_root = torch.empty(B, **i32)
    Bnd.heads(p, dev.h, None, dev.wstruct, logits, ref_tok, ref_val, ref_root, dev.ws)
    torch.cuda.synchronize()
    for call in range(2):                                     # two calls in a row
        tok = torch.full((B, K, 16), -7, **i32)
        val = torch.full((B, K, 16), float("nan"), device="cuda")
        root = torch.full((B,), -7, **i32)
        Bnd.heads_noalloc(p, dev.h, None, dev.wstruct, tok, val, root)
        torch.cuda.synchronize()
        for k in range(K):                                   # all 16 ranks, as medusa_heads
            np.testing.assert_array_equal(tok[:, k].cpu().numpy(), ref_tok[:, k].cpu().numpy())
            assert close(val[:, k].cpu().numpy(), ref_val[:, k].cpu().numpy(), ATOL, RTOL) <= 0
        np.testing.assert_array_equal(root.cpu().numpy(), ref_root.cpu().numpy())
    assert p.status() == 0


def test_noalloc_heads_carries_root_in():
    w = _mid()
    dev = setup(w)
    root_in = torch.tensor([5, 6, 7], dtype=torch.int32, device="cuda")
    tok = torch.empty(w.B, w.K, 16, dtype=torch.int32, device="cuda")
    val = torch.empty(w.B, w.K, 16, device="cuda")
    root = torch.empty(w.B, dtype=torch.int32, device="cuda")
    Bnd.heads_noalloc(dev.plan, dev.h, root_in, dev.wstruct, tok, val, root)
    torch.cuda.synchronize()
    assert root.tolist() == [5, 6, 7]


def test_noalloc_heads_batch8_full_vocab():
    # batch 8 of a 32000-token vocabulary: 8*5*32000*4 bytes of logits would not fit the
    # 4 MiB array, the fused top-k's candidate lists (8*5*250*128 bytes) do
    w = S.Workload("noalloc_b8", B=8, d=256, V=32000, Hq=4, Hkv=4, dh=64, K=4, dtype="bf16",
                   lengths=(5, 9, 17, 33, 65, 100, 120, 127), tree="greedy", s=(10, 10, 10, 10), N=30)
    test_noalloc_heads_matches_workspace_heads(w)


def test_noalloc_heads_rejects_plans_past_the_scratch_limit():
    # batch 64 of a 32000-token vocabulary: 64*5*250*128 bytes of candidate lists > 4 MiB
    p = Bnd.Plan(64, 256, 32000, 4, 4, 4, 64, Bnd.BF16, 64, (2, 2, 2, 2),
                 *Bnd.tree_cartesian((2, 2, 2, 2)))
    dummy = torch.zeros(64, dtype=torch.int32, device="cuda")
    with pytest.raises(Bnd.MedusaError) as e:
        Bnd.heads_noalloc(p, dummy, None, Bnd.weights_struct({}), dummy, dummy, dummy)
    assert e.value.code == Bnd.MEDUSA_ERR_UNSUPPORTED
