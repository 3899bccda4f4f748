"""GPU parity: every stage of the CUDA path against the fp64 oracle on the same seeded
inputs, called through the C ABI.  Sizes run from the tiny workload through ragged
multi-tile cases to the full Vicuna/Zephyr-shaped workloads (oracle on sampled
sequences where the batch is large)."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle as O
import synthetic as S
from medusa_head_speculative_gb300 import binding as Bnd

from harness import (Flagged, close, compare_sequence, oracle_step, record, run_stages, run_step,
                     setup)

pytestmark = pytest.mark.gpu


def _mid(**kw):
    """Ragged multi-tile bf16 case: GQA 8/2, vocab and rows not multiples of the tiles."""
    base = dict(name="mid", B=3, d=256, V=1000, Hq=8, Hkv=2, dh=64, K=4, dtype="bf16",
                lengths=(37, 100, 257), tree="greedy", s=(10, 10, 10, 10), N=30)
    base.update(kw)
    return S.Workload(**base)


_L13 = S.workload("vicuna13b").lengths
_SHORT13, _LONG13 = int(np.argmin(_L13)), int(np.argmax(_L13))

# name -> (workload, sampled sequences or None for all).  A sampled workload's other
# sequences still run on the GPU (and the fused step must equal the stages on them); the
# largest ones get their unsampled prefixes drawn on the device.
CASES = {
    "tiny": (S.workload("tiny"), None),
    "mid_greedy": (_mid(), None),
    "mid_typical": (_mid(mode="typical", temperature=0.7), None),
    "mid_paged": (_mid(page_size=16), None),
    "mid_b6_typical": (_mid(B=6, lengths=(1, 45, 64, 65, 130, 300), dh=128, Hq=4, Hkv=4,
                            mode="typical", temperature=1.3, s=(4, 3, 2, 2), tree="cartesian",
                            N=4 + 12 + 24 + 48), None),
    "mid_fp32_gqa": (_mid(dtype="f32", d=96, V=700, lengths=(5, 70, 33)), None),
    # fp32 batch of 6: the row-dot takes the activation rows in passes of 4, and every pass
    # keeps candidate lists of its own for the fused top-k
    "mid_fp32_b6": (_mid(dtype="f32", B=6, d=96, V=700, lengths=(3, 17, 40, 64, 90, 128)), None),
    # a vocabulary that is not a multiple of 4: scalar loads in the selection and the
    # verification statistics, ragged slices
    "mid_odd_vocab": (_mid(V=997, lengths=(12, 64, 129)), None),
    # the same at batch 1: the row-dot path, whose candidate slots are its CTAs' row ranges
    # (ragged against the heads' 997-row blocks)
    "mid_b1_odd_vocab": (_mid(B=1, V=997, lengths=(77,)), None),
    # 151 nodes of one query head per KV head: two 128-row attention tiles, three tree-key
    # chunks, ancestors across the tile boundary
    "mid_n150_mha": (_mid(B=2, Hq=4, Hkv=4, N=150, lengths=(70, 200)), None),
    "vicuna7b": (S.workload("vicuna7b"), None),
    "vicuna7b_typical": (S.workload("vicuna7b_typical"), None),
    # rejection sampling with seeded uniforms (mostly draws at the root on random weights)
    "mid_reject": (_mid(mode="reject", temperature=0.8), None),
    "vicuna7b_reject": (S.workload("vicuna7b", mode="reject", temperature=0.7), None),
    # four sampled sequences each, the 13B ones including its shortest and longest prefix
    "vicuna13b": (S.workload("vicuna13b"), tuple(sorted({0, 5, _SHORT13, _LONG13}))),
    "zephyr7b": (S.workload("zephyr7b"), (0, 3, 12, 15)),
    # the Vicuna-33B-shaped sweep: two sampled sequences per point, from the smallest to
    # the extreme corners (64 x 16K-token prefixes: the largest split counts and the
    # longest TMA walks; 64 x 129 nodes = 8256 node rows over many activation tiles)
    "vicuna33b_b4_l1024_n16": (S.vicuna33b(4, 1024, 16), (1, 2)),
    "vicuna33b_b16_l1024_n128": (S.vicuna33b(16, 1024, 128), (5, 11)),
    "vicuna33b_b64_l16384_n16": (S.vicuna33b(64, 16384, 16), (0, 63)),
    "vicuna33b_b64_l1024_n128": (S.vicuna33b(64, 1024, 128), (7, 40)),
}

# KV caches above this many bytes get only the sampled sequences' prefixes from the host
# streams; the rest are drawn on the device (sequences are independent, so they do not
# change the sampled sequences' outputs)
HOST_KV_LIMIT = 4 << 30


def _kv_bytes(w):
    return 2 * w.B * w.capacity * w.Hkv * w.dh * (4 if w.dtype == "f32" else 2)


def _compare(dev, g, seqs, root=None):
    """Compare the sampled sequences with the oracle; returns (compared, flagged)."""
    ow = O.oracle_weights(dev.cpu["wts"])
    compared, flagged = 0, []
    for b in seqs:
        r = oracle_step(dev, b, ow, root=None if root is None else int(root[b]))
        try:
            compare_sequence(g, r, b, dev.spec, dev.w, {}, root_given=root is not None)
            compared += 1
        except Flagged as e:
            flagged.append((b, str(e)))
    return compared, flagged


def _check(name):
    w, sample = CASES[name]
    seqs = list(sample) if sample else list(range(w.B))
    host_seqs = seqs if _kv_bytes(w) > HOST_KV_LIMIT else None
    dev = setup(w, host_seqs=host_seqs)
    g = run_stages(dev)
    compared, flagged = _compare(dev, g, seqs)
    if w.B == 1 and compared == 0:
        # the only sequence hit a near tie: a second seed, so that one is compared in full
        w2 = dataclasses.replace(w, seed=w.seed + 1)
        dev2 = setup(w2)
        c2, f2 = _compare(dev2, run_stages(dev2), seqs)
        compared += c2
        flagged += [(f"seed {w2.seed}", why) for _, why in f2]
        del dev2
    record(name, compared, flagged)
    assert compared >= max(1, len(seqs) - 1), flagged
    # the fused step equals the chained stages exactly, and compacts the cache
    len_out = torch.empty_like(dev.length)
    s = run_step(dev, len_out=len_out)
    np.testing.assert_array_equal(s["out_tok"], g["out_tok"])
    np.testing.assert_array_equal(s["n_acc"], g["n_acc"])
    np.testing.assert_array_equal(s["path"], g["path"])
    np.testing.assert_array_equal(s["root_next"].cpu().numpy(), g["root_next"])
    np.testing.assert_array_equal(s["h_next"].cpu().numpy(), g["h_next"])
    np.testing.assert_array_equal(s["len_out"], np.array(w.lengths) + g["n_acc"])
    assert dev.plan.status() == 0
    for b in range(w.B):
        L, n = w.lengths[b], int(g["n_acc"][b])
        kc = _seq_cache(dev, dev.kc, b, L, L + n)
        vc = _seq_cache(dev, dev.vc, b, L, L + n)
        for l in range(n):
            node = g["path"][b, l]
            np.testing.assert_array_equal(kc[l], g["tk"][b, node])
            np.testing.assert_array_equal(vc[l], g["tv"][b, node])
        if host_seqs is None or b in host_seqs:
            k0, _ = S.kv_prefix(w, b)                                   # prefix untouched
            np.testing.assert_array_equal(_seq_cache(dev, dev.kc, b, 0, L), k0.float().numpy())
        assert not _seq_cache_any(dev, dev.kc, b, L + n)                 # nothing past the path
    return g, flagged


def _seq_rows(dev, t, b, t0, t1):
    """Logical cache rows t0..t1-1 of sequence b as a device tensor (pages resolved)."""
    w = dev.w
    if not w.page_size:
        return t[b, t0:t1]
    slots = torch.arange(t0, t1, device=t.device)
    pages = dev.pt[b].long()[slots // w.page_size]
    return t[pages, slots % w.page_size]


def _seq_cache(dev, t, b, t0, t1):
    return _seq_rows(dev, t, b, t0, t1).float().cpu().numpy()


def _seq_cache_any(dev, t, b, t0):
    return bool(_seq_rows(dev, t, b, t0, dev.w.capacity).any())


@pytest.mark.parametrize("name", list(CASES))
def test_step_matches_oracle(name):
    _check(name)


@pytest.mark.parametrize("name", ["mid_greedy", "mid_b6_typical", "vicuna7b"])
def test_step_with_given_root(name):
    """A root carried in from the previous step (the LM head pass on h_t is skipped): the
    stages and the fused step both match the oracle's step with that root."""
    w, sample = CASES[name]
    dev = setup(w)
    rng = np.random.default_rng(11)
    roots = rng.integers(0, w.V, size=w.B).astype(np.int32)
    root_in = torch.from_numpy(roots).cuda()
    g = run_stages(dev, root_in=root_in)
    np.testing.assert_array_equal(g["root"], roots)
    seqs = list(sample) if sample else list(range(w.B))
    compared, flagged = _compare(dev, g, seqs, root=roots)
    if w.B == 1 and compared == 0:
        dev2 = setup(dataclasses.replace(w, seed=w.seed + 1))
        c2, f2 = _compare(dev2, run_stages(dev2, root_in=root_in), seqs, root=roots)
        compared += c2
        flagged += [(f"seed {w.seed + 1}", why) for _, why in f2]
        del dev2
    record(f"given_root_{name}", compared, flagged)
    assert compared >= max(1, len(seqs) - 1), flagged
    s = run_step(dev, root_in=root_in, len_out=torch.empty_like(dev.length))
    np.testing.assert_array_equal(s["out_tok"], g["out_tok"])
    np.testing.assert_array_equal(s["path"], g["path"])
    np.testing.assert_array_equal(s["h_next"].cpu().numpy(), g["h_next"])
    assert dev.plan.status() == 0


def test_fp32_tiny_tight_tolerance():
    w = S.workload("tiny")
    dev = setup(w)
    g = run_stages(dev)
    r = oracle_step(dev, 0)
    assert close(g["logits"][0, 0], r.z0, 2e-5, 1e-5) <= 0
    assert close(g["o"][0], r.o, 2e-5, 1e-5) <= 0
    assert close(g["vlog"][0], r.zv, 5e-5, 1e-5) <= 0


def test_generate_loop_matches_sequential_greedy():
    """Steps chained on the GPU (root_next and h_next carried, cache compacted in place)
    emit the same tokens as the oracle's Medusa loop and plain greedy decoding."""
    w = S.workload("tiny")
    wts = S.planted_weights(w)
    h0 = wts["emb"][7].float().unsqueeze(0).clone()
    dev = setup(w, wts_cpu=wts, h_cpu=h0)
    ow = O.oracle_weights(wts)
    dims = {"Hq": w.Hq, "Hkv": w.Hkv, "dh": w.dh, "rope_base": w.rope_base}
    k0, v0 = S.kv_prefix(w, 0)
    steps = 8
    toks_o, steps_o, kc_o, vc_o = O.medusa_generate(ow, h0[0], k0, v0, dev.spec, dims,
                                                    {"mode": "greedy"}, steps)
    seq, _, _ = O.sequential_greedy(ow, h0[0], k0, v0, dims, len(toks_o))
    assert toks_o == seq
    toks_g, root = [], None
    for _ in range(steps):
        s = run_step(dev, root_in=root)
        n = int(s["n_acc"][0])
        toks_g += list(s["out_tok"][0, :n])
        dev.h = s["h_next"]
        root = s["root_next"]
    assert toks_g == toks_o
    assert int(dev.length[0]) == kc_o.shape[0]
    kc = dev.kc[0, :kc_o.shape[0]].float().cpu().numpy()
    assert close(kc, kc_o, 1e-4, 1e-4) <= 0
    assert max(s_.m for s_ in steps_o) >= 2


def test_exact_ties_take_the_lowest_token_id():
    """Duplicated LM-head / head rows give bitwise-equal logits: the lowest id wins."""
    w = S.workload("tiny")
    wts = S.head_init_weights(S.weights(w))
    lm = wts["lm"].clone()
    h = S.hidden(w)
    z = lm.double() @ h[0].double()
    best = int(torch.argmax(z))
    dup = best - 5 if best >= 5 else best + 5
    lm[dup] = lm[best]                   # an exact copy of the best row
    lo, hi = min(dup, best), max(dup, best)
    wts["lm"] = lm
    wts["w2"] = lm.unsqueeze(0).expand_as(wts["w2"]).contiguous()
    dev = setup(w, wts_cpu=wts, h_cpu=h)
    g = run_stages(dev)
    assert g["logits"][0, 0, lo] == g["logits"][0, 0, hi]
    assert g["root"][0] == lo
    assert g["topk_tok"][0, 0, 0] == lo and g["topk_tok"][0, 0, 1] == hi


def test_root_only_tree_and_empty_prefix():
    w = S.Workload("root_only", B=2, d=128, V=512, Hq=4, Hkv=2, dh=32, K=1, dtype="bf16",
                   lengths=(0, 9), tree="greedy", s=(3,), N=0)
    dev = setup(w)
    g = run_stages(dev)
    for b in range(2):
        compare_sequence(g, oracle_step(dev, b), b, dev.spec, w, {})


def test_typical_at_temperature_zero_is_greedy():
    wg = _mid()
    wt = dataclasses.replace(wg, mode="typical", temperature=0.0)
    g1 = run_stages(setup(wg))
    g2 = run_stages(setup(wt))
    np.testing.assert_array_equal(g1["out_tok"], g2["out_tok"])
    np.testing.assert_array_equal(g1["n_acc"], g2["n_acc"])


def test_capacity_overflow_sets_flag_and_clamps():
    w = dataclasses.replace(S.workload("tiny"), reserve=0)     # capacity = 64 = prefix
    dev = setup(w)
    len_out = torch.empty_like(dev.length)
    run_step(dev, len_out=len_out)
    assert dev.plan.status() & Bnd.FLAG_KV_CAPACITY
    assert int(len_out[0]) == w.capacity
    assert dev.plan.status() == 0                               # reading clears the word


def test_page_out_of_range_sets_flag():
    w = _mid(page_size=16)
    dev = setup(w)
    dev.pt[1, 0] = 10 ** 6                                      # checked before any access
    run_stages(dev)
    assert dev.plan.status() & Bnd.FLAG_PAGE_RANGE


def test_workspace_too_small_is_rejected():
    dev = setup(S.workload("tiny"))
    dev.ws = dev.ws[:-256]
    with pytest.raises(Bnd.MedusaError) as e:
        run_step(dev)
    assert e.value.code == Bnd.MEDUSA_ERR_WORKSPACE


def test_nonfinite_hidden_state_is_contained_and_flagged():
    """A NaN in one sequence's h_t never faults: its candidate tokens come out of range and
    are flagged (then clamped), and the other sequences' outputs are unchanged."""
    w = _mid()
    dev = setup(w)
    clean = run_step(dev, len_out=torch.empty_like(dev.length))
    assert dev.plan.status() == 0
    dev.h[0, 5] = float("nan")
    bad = run_step(dev, len_out=torch.empty_like(dev.length))
    assert dev.plan.status() & (Bnd.FLAG_TOKEN_RANGE | Bnd.FLAG_NONFINITE)
    np.testing.assert_array_equal(bad["out_tok"][1:], clean["out_tok"][1:])
    np.testing.assert_array_equal(bad["path"][1:], clean["path"][1:])
    np.testing.assert_array_equal(bad["h_next"][1:].cpu().numpy(), clean["h_next"][1:].cpu().numpy())
    assert ((bad["out_tok"][0] >= -1) & (bad["out_tok"][0] < w.V)).all()


def _guarded(n, dtype, fill):
    """A flat buffer of n elements with 4096-element guard bands filled with `fill`."""
    G = 4096
    big = torch.full((n + 2 * G,), fill, dtype=dtype, device="cuda")
    return big, big[G:G + n]


def test_step_writes_stay_inside_the_buffers():
    """Canary bands around every buffer the step writes (outputs, lengths, workspace) stay
    intact, and the inputs it only reads (h_t, the cached prefix) are unchanged."""
    for w in (_mid(page_size=16), _mid(B=2, Hq=4, Hkv=4, N=150, lengths=(70, 200)), S.workload("tiny")):
        dev = setup(w)
        B, K, d = w.B, w.K, w.d
        i32 = torch.int32
        canary = {}
        def buf(name, shape, dtype, fill):
            n = int(np.prod(shape))
            big, mid = _guarded(n, dtype, fill)
            canary[name] = (big, n, fill)
            return mid.view(shape)
        out_tok = buf("out_tok", (B, K + 1), i32, -12345)
        n_acc = buf("n_acc", (B,), i32, -12345)
        path = buf("path", (B, K + 1), i32, -12345)
        h_next = buf("h_next", (B, d), torch.float32, 1234.5)
        root_next = buf("root_next", (B,), i32, -12345)
        len_out = buf("len_out", (B,), i32, -12345)
        ws = buf("ws", (dev.plan.workspace_size,), torch.uint8, 0xA5)
        h0 = dev.h.clone()
        k0 = dev.kc.clone()
        kv = Bnd.kv_struct(dev.kc, dev.vc, dev.length, len_out, dev.pt)
        outs = Bnd.outputs_struct(out_tok, n_acc, path, h_next, root_next)
        from harness import accept_of
        Bnd.step(dev.plan, dev.h, None, dev.wstruct, kv, Bnd.accept_struct(**accept_of(w)), outs, ws)
        torch.cuda.synchronize()
        assert dev.plan.status() == 0
        G = 4096
        for name, (big, n, fill) in canary.items():
            lo, hi = big[:G], big[G + n:]
            ref = torch.full_like(lo, fill)
            assert torch.equal(lo, ref) and torch.equal(hi, ref), f"{w.name}: {name} guard band written"
        assert torch.equal(dev.h, h0)
        # the cache changes only in the slots after each prefix (the compacted path)
        kc = dev.kc.float().cpu()
        kref = k0.float().cpu()
        if not w.page_size:
            for b in range(B):
                L = w.lengths[b]
                assert torch.equal(kc[b, :L], kref[b, :L])
                assert torch.equal(kc[b, L + int(n_acc[b]):], kref[b, L + int(n_acc[b]):])


def test_reject_on_planted_tiny_model_follows_the_oracle_over_steps():
    """Rejection sampling on a model whose heads are usually right: candidates are accepted
    and the walk goes deep; each step (fresh uniforms) matches the oracle's."""
    import dataclasses as dc
    w = dc.replace(S.workload("tiny"), mode="reject", temperature=1.0)
    wts = S.planted_weights(w)
    h0 = wts["emb"][7].float().unsqueeze(0).clone()
    dev = setup(w, wts_cpu=wts, h_cpu=h0)
    ow = O.oracle_weights(wts)
    dims = {"Hq": w.Hq, "Hkv": w.Hkv, "dh": w.dh, "rope_base": w.rope_base}
    k, v = S.kv_prefix(w, 0)
    k, v = k.double().numpy(), v.double().numpy()
    h = h0[0].double().numpy()
    root = None
    deepest = 0
    for step in range(6):
        dev.uni = S.uniforms(w, step).cuda()
        acc = {"mode": "reject", "temperature": 1.0, "eps": w.eps, "delta": w.delta,
               "uniforms": S.uniforms(w, step)[0].numpy().astype(np.float64)}
        r = O.medusa_step(ow, h, k, v, dev.spec, dims, acc,
                          root=None if root is None else int(root[0]), s=list(w.s))
        g = run_step(dev, root_in=root)
        gm = int(g["n_acc"][0]) - 1
        if r.rs_margin >= O.NEAR_P:
            assert list(g["path"][0, :gm + 1]) == list(r.path_nodes), step
            assert int(g["root_next"][0]) == r.root_next, step
        else:
            break
        deepest = max(deepest, gm)
        # carry the state: the cache grows by the kept nodes' keys/values (oracle side)
        k = np.concatenate([k, r.kv_new[0]])
        v = np.concatenate([v, r.kv_new[1]])
        h = r.h_next
        dev.h = g["h_next"]
        root = g["root_next"]
    assert deepest >= 1
    assert dev.plan.status() == 0


def test_reject_at_temperature_zero_is_greedy():
    import dataclasses as dc
    wg = _mid()
    wr = dc.replace(wg, mode="reject", temperature=0.0)
    g1 = run_stages(setup(wg))
    g2 = run_stages(setup(wr))
    np.testing.assert_array_equal(g1["out_tok"], g2["out_tok"])
    np.testing.assert_array_equal(g1["root_next"], g2["root_next"])


def test_loop_rejects_rejection_sampling():
    import dataclasses as dc
    from harness import accept_of
    w = dc.replace(_mid(), mode="reject", temperature=0.8)
    dev = setup(w)
    root = torch.zeros(w.B, dtype=torch.int32, device="cuda")
    kv = Bnd.kv_struct(dev.kc, dev.vc, dev.length, dev.length, dev.pt)
    tokens = torch.empty(2, w.B, w.K + 1, dtype=torch.int32, device="cuda")
    n_acc = torch.empty(2, w.B, dtype=torch.int32, device="cuda")
    with pytest.raises(Bnd.MedusaError) as e:
        Bnd.Loop(dev.plan, dev.wstruct, kv, Bnd.accept_struct(**accept_of(w, dev)), dev.h, root,
                 tokens, n_acc, dev.ws)
    assert e.value.code == Bnd.MEDUSA_ERR_UNSUPPORTED
