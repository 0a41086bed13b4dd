"""Pins of the oracle's two-level NVFP4 scale (per-tensor encode scale g times the
per-16 E4M3 scales; the pages' input_global_scale and "alpha = igs * global_sf").

What fixes it other than the oracle itself:
* closed forms of g = fp32(2688 / amax);
* with g a power of two, two-level quantisation is one-level quantisation of
  the exactly scaled input, and dequantisation divides exactly;
* the block holding the tensor's amax lands on the top E4M3 scale (448);
* the dequantised error stays within 1.25 * dec(scale) / g per element (the
  largest half-step detour of the two-stage E2M1 rule: 5.25 -> 4);
* the purpose the pages give it: small-magnitude weights no longer get
  subnormal block scales;
* with every encode scale a power of two, the whole two-level FFN equals the
  one-level FFN bit for bit (a dropped or inverted alpha factor would scale the
  output by that power of two).
"""
import numpy as np
import pytest

import inputs
from oracle import moe as omoe
from oracle import nvfp4 as onv


def test_global_scale_closed_forms():
    def g(vals):
        return onv.global_scale(np.array([vals], dtype=np.float32))

    assert g([0.0, -2688.0]) == np.float32(1.0)
    assert g([1344.0, 1.0]) == np.float32(2.0)
    assert g([448.0]) == np.float32(6.0)
    assert g([-3.0, 2.0]) == np.float32(896.0)
    assert g([0.0, 0.0]) == np.float32(1.0)                 # all-zero tensor
    assert g([1e-38]) == np.float32(1.0)                    # quotient not finite in fp32
    assert g([7.0]) == np.float32(np.float32(2688.0) / np.float32(7.0))


@pytest.mark.parametrize("k", [-3, 0, 5, 11])
def test_power_of_two_scale_is_exact_scaling(k):
    rng = np.random.default_rng(40 + k)
    x = rng.standard_normal((64, 256)).astype(np.float32)
    g = np.float32(2.0 ** k)
    q2, sf2 = onv.quantize_rows(x, g)
    q1, sf1 = onv.quantize_rows((x * g).astype(np.float32))
    assert np.array_equal(q1, q2) and np.array_equal(sf1, sf2)
    assert np.array_equal(onv.dequantize_rows(q2, sf2, g), onv.dequantize_rows(q2, sf2) / 2.0 ** k)


def test_amax_block_lands_on_top_scale_and_error_bound():
    rng = np.random.default_rng(3)
    x = (rng.standard_t(3, size=(128, 512)) * 0.7).astype(np.float32)
    g = onv.global_scale(x)
    q, sf = onv.quantize_rows(x, g)
    r, c = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    assert sf[r, c // 16] == 0x7E
    assert sf.max() <= 0x7E
    dq = onv.dequantize_rows(q, sf, g)
    d = onv.E4M3_TABLE_F32[sf].astype(np.float64) / np.float64(g)
    normal = ((sf >> 3) & 0xF) > 0
    err = np.abs(dq - x).reshape(128, 32, 16).max(axis=2)
    assert np.all(err[normal] <= 1.25 * d[normal] * (1 + 1e-12))


def test_two_level_removes_subnormal_weight_scales():
    w = (np.random.default_rng(5).standard_normal((256, 1024)) * 0.02).astype(np.float32)
    _, sf1 = onv.quantize_rows(w)
    _, sf2 = onv.quantize_rows(w, onv.global_scale(w))
    subnormal = lambda sf: np.mean(((sf >> 3) & 0xF) == 0)
    assert subnormal(sf1) > 0.9            # one level: almost every block subnormal
    assert subnormal(sf2) == 0.0           # two levels: none


def test_two_level_ffn_equals_one_level_with_power_of_two_scales():
    spec = inputs.moe_spec(T=96, H=256, I=256, E=4, top_k=2, seed=44)
    x_t, x = inputs.moe_x(spec)
    x = np.clip(x, -4.0, 4.0)
    x[0, 0] = 5.25                          # amax 2688 / 512 -> g_x = 512
    logits = inputs.moe_logits(spec)
    rng = np.random.default_rng(45)
    E, H, I = spec["E"], spec["H"], spec["I"]
    w1 = np.clip(rng.standard_normal((E, 2 * I, H)) * 0.5, -2.5, 2.5).astype(np.float32)
    w2 = np.clip(rng.standard_normal((E, H, I)) * 0.5, -2.5, 2.5).astype(np.float32)
    w1[:, 0, 0] = 2.625                     # amax 2688 / 1024 -> g = 1024
    w2[:, 0, 0] = -2.625
    gs = omoe.two_level_scales(x, w1, w2)
    assert gs["x"] == 512 and np.all(gs["w1"] == 1024) and np.all(gs["w2"] == 1024)
    one = omoe.moe_ffn(x, logits, w1, w2, spec["top_k"])
    two = omoe.moe_ffn(x, logits, w1, w2, spec["top_k"], a2_gscale=np.float32(4.0))
    # the scale codes moved by exact powers of two; every dequantised operand and
    # every output is the same
    assert np.array_equal(one["a1_q"], two["a1_q"]) and np.array_equal(one["w1_q"], two["w1_q"])
    assert not np.array_equal(one["a1_sf"], two["a1_sf"])
    assert np.array_equal(one["g_full"], two["g_full"])
    assert np.array_equal(one["h"], two["h"])
    assert np.array_equal(one["rows"], two["rows"])
    assert np.array_equal(one["y"], two["y"])


def test_two_level_tokens_path_matches_batch_path():
    spec = inputs.moe_spec(T=40, H=256, I=256, E=6, top_k=2, seed=46)
    x_t, x = inputs.moe_x(spec)
    logits = inputs.moe_logits(spec)
    w1, w2 = inputs.moe_all_weights(spec)
    a2g = np.float32(37.5)
    full = omoe.moe_ffn(x, logits, w1, w2, spec["top_k"], a2_gscale=a2g)
    pick = np.array([0, 7, 39])
    tok = omoe.moe_ffn_tokens(x[pick], logits[pick], lambda e: w1[e], lambda e: w2[e], spec["top_k"],
                              two_level=dict(x=full["gscales"]["x"], a2=a2g))
    assert np.array_equal(tok["y"], full["y"][pick])
    rows = full["inv_perm"][pick].ravel()
    assert np.array_equal(tok["a2_q"].reshape(len(rows), -1), full["a2_q"][rows])
