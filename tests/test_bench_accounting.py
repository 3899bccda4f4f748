"""The byte and FLOP accounting behind bench.py's roofline (CPU only).

Every weight matrix of a step is counted once across the per-kernel figures, whichever
launch reads it: at batch 1 the LM head's root pass shares the first heads launch, from
batch 2 it is part of the vocabulary launch.  The per-kernel weight bytes must then add up
to the step's weight bytes, and moving the root pass between launches must change no
total."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synthetic as S  # noqa: E402


def _weights_only(w, n1, tc):
    """Per-kernel bytes with every activation, output and cache term removed."""
    kb = bench.kernel_bytes(w, n1, tc)
    es = 4 if w.dtype == "f32" else 2
    B = w.B
    K, d, V = w.K, w.d, w.V
    M = B * n1
    qd, kd = w.Hq * w.dh, w.Hkv * w.dh
    act = 4 if tc else 0
    heads_w1 = kb["heads_w1"] - (B * d * 4 + B * K * d * (4 + act) + (0 if tc else B * V * 4))
    heads_vocab = kb["heads_vocab"] - (B * (K + (1 if tc else 0)) * (d * 4 + V * 4))
    qkv = kb["layer_qkv"] - (M * d * 2 + M * (qd + 2 * kd) * 4)
    out = kb["layer_out"] - (M * qd * 4 + M * d * 10)
    verify = kb["verify_logits"] - (M * d * 4 + M * V * 4)
    return heads_w1, heads_vocab, qkv, out, verify, es


@pytest.mark.parametrize("name", ["tiny", "vicuna7b", "vicuna13b", "zephyr7b"])
@pytest.mark.parametrize("tc", [False, True])
def test_each_weight_matrix_is_counted_once(name, tc):
    w = S.workload(name)
    n1 = 22 if name == "tiny" else 65
    w1, vocab, qkv, out, verify, es = _weights_only(w, n1, tc)
    K, d, V = w.K, w.d, w.V
    qd, kd = w.Hq * w.dh, w.Hkv * w.dh
    # the heads' two launches read W1, W2 and the LM head (root pass) exactly once
    assert w1 + vocab == (K * d * d + K * V * d + V * d) * es
    assert w1 == (K * d * d + (0 if tc else V * d)) * es
    assert qkv == (qd + 2 * kd) * d * es
    assert out == d * qd * es
    assert verify == V * d * es


@pytest.mark.parametrize("name", ["vicuna7b", "vicuna13b"])
def test_root_pass_moves_flops_between_launches_not_the_total(name):
    w = S.workload(name)
    a = bench.kernel_flops(w, 65, True)
    b = bench.kernel_flops(w, 65, False)
    assert a["heads_w1"] + a["heads_vocab"] == b["heads_w1"] + b["heads_vocab"]
    assert b["heads_w1"] - a["heads_w1"] == 2 * w.B * w.V * w.d
    assert {k: v for k, v in a.items() if not k.startswith("heads")} == \
           {k: v for k, v in b.items() if not k.startswith("heads")}


def test_step_bytes_cover_the_kernels_weights():
    w = S.workload("vicuna7b")
    n1 = 65
    w1, vocab, qkv, out, verify, es = _weights_only(w, n1, False)
    sb = bench.step_bytes(w, n1)
    kv = sum(w.lengths) * 2 * w.Hkv * w.dh * es + w.B * n1 * 2 * w.Hkv * w.dh * es * 2
    gather = w.B * n1 * w.d * es
    assert sb == w1 + vocab + qkv + out + verify + kv + gather
