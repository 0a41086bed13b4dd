"""Pins of the oracle's shared expert (a dense FFN of every token, added after
the routed slots before the one BF16 rounding).

* closed form: the shared expert equals the routed path with a single expert,
  top-1 (its softmax weight is exactly 1), on the same weights -- bit for bit;
* zero shared weights leave the routed output unchanged;
* additivity: with a shared row that is exact in BF16 and small integer-valued
  routed rows, y is the exact sum;
* the per-token path equals the batch path with the shared expert.
"""
import numpy as np

import inputs
from oracle import moe as omoe


def _small():
    spec = inputs.moe_spec(T=70, H=256, I=256, E=4, top_k=2, seed=80)
    _, x = inputs.moe_x(spec)
    logits = inputs.moe_logits(spec)
    w1, w2 = inputs.moe_all_weights(spec)
    w1s, w2s = inputs.moe_shared_weights(spec)
    return spec, x, logits, w1, w2, w1s, w2s


def test_shared_expert_is_a_single_routed_expert():
    spec, x, _, _, _, w1s, w2s = _small()
    sh = omoe.shared_expert_rows(x, w1s, w2s)
    one = omoe.moe_ffn(x, np.zeros((spec["T"], 1), np.float32), w1s[None], w2s[None], 1)
    assert np.all(one["w"] == 1.0)
    assert np.array_equal(sh["rows"], one["y"])
    assert np.array_equal(sh["h"], one["h"][one["inv_perm"][:, 0]])


def test_zero_shared_expert_changes_nothing():
    spec, x, logits, w1, w2, w1s, w2s = _small()
    plain = omoe.moe_ffn(x, logits, w1, w2, spec["top_k"])
    zero = omoe.moe_ffn(x, logits, w1, w2, spec["top_k"], shared=(0 * w1s, 0 * w2s))
    assert not np.any(zero["shared"]["rows"])
    assert np.array_equal(plain["y"], zero["y"])


def test_combine_adds_the_shared_row_last():
    rows = np.array([[1.0, 2.0], [3.0, -4.0], [0.5, 0.5]], dtype=np.float64)
    inv = np.array([[1, 0], [2, 1]])
    w = np.array([[0.5, 0.5], [1.0, 0.0]], dtype=np.float32)
    shared = np.array([[10.0, -1.0], [0.0, 96.0]])
    y = omoe.combine(rows, inv, w, shared)
    assert np.array_equal(y, np.array([[12.0, -2.0], [0.5, 96.5]]))   # all exact in BF16


def test_tokens_path_matches_batch_path_with_shared_expert():
    spec, x, logits, w1, w2, w1s, w2s = _small()
    full = omoe.moe_ffn(x, logits, w1, w2, spec["top_k"], shared=(w1s, w2s))
    pick = np.array([0, 33, 69])
    tok = omoe.moe_ffn_tokens(x[pick], logits[pick], lambda e: w1[e], lambda e: w2[e], spec["top_k"],
                              shared=(w1s, w2s))
    assert np.array_equal(tok["y"], full["y"][pick])
