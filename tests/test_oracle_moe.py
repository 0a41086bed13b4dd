"""Pins for the oracle's routing, permutation, GEMMs, SwiGLU epilogue and combine
(CPU only): brute force on tiny inputs, library routines, invariants, and
special cases that reduce to a textbook result."""
import numpy as np
import pytest
import scipy.special
import torch

import inputs
from oracle import moe, nvfp4


# ----------------------------------------------------------------- BF16 --
def test_round_to_bf16_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000)),
                        [0.0, 1.0, -1.0, 1.00390625, 1.01171875]])
    # torch rounds from fp32; use values exactly representable in fp32 so the
    # single rounding to BF16 is the same rounding
    x32 = x.astype(np.float32)
    ref = torch.from_numpy(x32).to(torch.bfloat16).float().numpy()
    assert np.array_equal(moe.round_to_bf16(x32.astype(np.float64)).astype(np.float32), ref)
    bits = moe.bf16_bits(ref)
    assert np.array_equal(moe.bf16_from_bits(bits), ref)


# -------------------------------------------------------------- routing --
def test_route_topk_brute_force():
    rng = np.random.default_rng(1)
    logits = rng.standard_normal((50, 16)).astype(np.float32)
    logits[3, 5] = logits[3, 9] = logits[3].max() + 1      # an exact tie at the top
    logits[4, :] = 0.5                                       # all equal
    ids, w = moe.route_topk(logits, 4)
    for t in range(50):
        ref = sorted(range(16), key=lambda e: (-float(logits[t, e]), e))[:4]
        assert list(ids[t]) == ref
        sel = logits[t, ref].astype(np.float64)
        assert np.allclose(w[t], scipy.special.softmax(sel), rtol=1e-14, atol=0)
    assert list(ids[3][:2]) == [5, 9]
    assert list(ids[4]) == [0, 1, 2, 3]
    assert np.allclose(w.sum(1), 1.0)


def test_permute_invariants_and_brute_force():
    rng = np.random.default_rng(2)
    T, E, k = 300, 6, 3
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    p = moe.permute(ids, E)
    counts, offs, perm, inv = p["counts"], p["offsets"], p["perm_token"], p["inv_perm"]
    assert counts.sum() == T * k
    assert np.all(offs % 128 == 0) and offs[0] == 0
    assert np.all(np.diff(offs) >= counts) and np.all(np.diff(offs) - counts < 128)
    for t in range(T):
        for j in range(k):
            r = inv[t, j]
            assert perm[r] == t and offs[ids[t, j]] <= r < offs[ids[t, j] + 1]
    for e in range(E):
        rows = perm[offs[e]:offs[e + 1]]
        real = rows[:counts[e]]
        assert np.all(np.diff(real) > 0)                      # ascending tokens
        assert np.all(rows[counts[e]:] == -1)
        assert list(real) == [t for t in range(T) if e in ids[t]]


def test_stage_activation_rows():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((10, 64)).astype(np.float32)
    perm = np.array([3, -1, 0, 9, -1], np.int64)
    q, sf = moe.stage_activation(x, perm)
    xq, xsf = nvfp4.quantize_rows(x)
    assert np.array_equal(q[0], xq[3]) and np.array_equal(q[3], xq[9])
    assert not q[1].any() and not sf[4].any()


# ---------------------------------------------------------------- GEMMs --
def test_grouped_gemm_triple_loop():
    rng = np.random.default_rng(4)
    offs = np.array([0, 3, 3, 8])
    a = rng.standard_normal((8, 5))
    b = rng.standard_normal((3, 4, 5))
    out = moe.grouped_gemm(a, offs, b, alpha=0.5)
    for r in range(8):
        e = int(np.searchsorted(offs, r, side="right") - 1)
        for n in range(4):
            acc = 0.0
            for kk in range(5):
                acc += a[r, kk] * b[e, n, kk]
            assert abs(out[r, n] - 0.5 * acc) < 1e-12


def test_dequantize_matches_scalar_decoders_and_nibble_order():
    q = np.array([[0x21, 0xF7]], np.uint8)            # nibbles 1,2,7,F
    sf = np.array([[0x38]], np.uint8)                   # scale 1.0
    q = np.pad(q, ((0, 0), (0, 6)))
    dq = nvfp4.dequantize_rows(q, sf)
    assert list(dq[0, :4]) == [0.5, 1.0, 6.0, -6.0]
    rng = np.random.default_rng(5)
    q = rng.integers(0, 256, (3, 16), dtype=np.uint8)
    sf = rng.integers(0x20, 0x50, (3, 2), dtype=np.uint8)
    dq = nvfp4.dequantize_rows(q, sf)
    for r in range(3):
        for c in range(32):
            byte = int(q[r, c // 2])
            nib = byte & 0xF if c % 2 == 0 else byte >> 4
            assert dq[r, c] == nvfp4.e2m1_decode(nib) * nvfp4.e4m3_decode(int(sf[r, c // 16]))


def test_one_hot_gemm_locates_products():
    # one nonzero nibble in A (row 2, element 37) and one in B (row 5, element 37)
    K = 64
    a_q = np.zeros((4, K // 2), np.uint8)
    b_q = np.zeros((8, K // 2), np.uint8)
    a_q[2, 18] = 0x30          # element 37 -> high nibble of byte 18, code 3 (1.5)
    b_q[5, 18] = 0x70          # code 7 (6.0)
    a_sf = np.full((4, K // 16), 0x38, np.uint8)
    b_sf = np.full((8, K // 16), 0x38, np.uint8)
    a_sf[2, 2] = 0x40          # 2.0 on the block of element 37
    b_sf[5, 2] = 0x30          # 0.5
    out = moe.grouped_gemm(nvfp4.dequantize_rows(a_q, a_sf), np.array([0, 4]),
                           nvfp4.dequantize_rows(b_q, b_sf)[None])
    expect = np.zeros((4, 8))
    expect[2, 5] = 1.5 * 2.0 * 6.0 * 0.5
    assert np.array_equal(out, expect)


# -------------------------------------------------------------- combine --
def test_combine_brute_force():
    rng = np.random.default_rng(6)
    rows = moe.round_to_bf16(rng.standard_normal((20, 8)))
    inv = rng.integers(0, 20, (5, 3))
    w = rng.random((5, 3))
    y = moe.combine(rows, inv, w)
    for t in range(5):
        for c in range(8):
            acc = 0.0
            for j in range(3):
                acc += w[t, j] * rows[inv[t, j], c]
            assert y[t, c] == moe.round_to_bf16(np.array([acc]))[0]


# ------------------------------------------------------ whole-path checks --
def test_moe_ffn_single_expert_reduces_to_dense_chain():
    """E=1, k=1: routing weight 1, one group: y = bf16(L2(requant(swiglu(L1(x)))))."""
    spec = inputs.moe_spec(T=40, H=128, I=64, E=1, top_k=1, seed=3)
    _, x = inputs.moe_x(spec)
    w1, w2 = inputs.moe_all_weights(spec)
    out = moe.moe_ffn(x, inputs.moe_logits(spec), w1, w2, 1)
    assert np.all(out["w"] == 1.0) and out["offsets"].tolist() == [0, 128]
    xq, xsf = nvfp4.quantize_rows(x)
    w1q, w1sf = nvfp4.quantize_rows(w1[0])
    g = nvfp4.dequantize_rows(xq, xsf) @ nvfp4.dequantize_rows(w1q, w1sf).T
    gate, up = nvfp4.deinterleave_gu8(g)
    h = (gate * scipy.special.expit(gate) * up).astype(np.float32)
    assert np.allclose(h, out["h"][:40], rtol=1e-6, atol=1e-30)
    q2, sf2 = nvfp4.quantize_rows(out["h"][:40])
    w2q, w2sf = nvfp4.quantize_rows(w2[0])
    o = nvfp4.dequantize_rows(q2, sf2) @ nvfp4.dequantize_rows(w2q, w2sf).T
    assert np.array_equal(out["y"], moe.round_to_bf16(o))


def test_moe_ffn_large_gate_makes_swiglu_linear_in_up():
    """Gate rows scaled so g >> 0 everywhere: silu(g) ~= g, h ~= g * u."""
    spec = inputs.moe_spec(T=16, H=128, I=32, E=2, top_k=1, seed=5)
    _, x = inputs.moe_x(spec)
    x = np.abs(x)
    w1, w2 = inputs.moe_all_weights(spec)
    g_rows = w1.reshape(2, 32 // 8, 2, 8, 128)
    g_rows[:, :, 0] = np.abs(g_rows[:, :, 0]) * 50
    out = moe.moe_ffn(x, inputs.moe_logits(spec), w1, w2, 1)
    g, u = nvfp4.deinterleave_gu8(out["g_full"])
    real = out["perm_token"] >= 0
    assert np.all(g[real] > 20)
    assert np.allclose(out["h"][real], (g * u)[real], rtol=1e-6)


def test_moe_ffn_tiny_config_runs_and_is_consistent():
    spec = dict(inputs.CONFIGS["tiny"])
    _, x = inputs.moe_x(spec)
    w1, w2 = inputs.moe_all_weights(spec)
    out = moe.moe_ffn(x, inputs.moe_logits(spec), w1, w2, spec["top_k"])
    assert out["y"].shape == (128, 512)
    assert np.isfinite(out["y"]).all()
    # the combined output is the weighted sum of each token's expert rows
    t = 7
    acc = sum(out["w"][t, j] * out["rows"][out["inv_perm"][t, j]] for j in range(2))
    assert np.array_equal(out["y"][t], moe.round_to_bf16(acc))


def test_per_token_path_equals_whole_batch():
    spec = inputs.moe_spec(T=50, H=256, I=256, E=4, top_k=2, seed=12)
    _, x = inputs.moe_x(spec)
    w1, w2 = inputs.moe_all_weights(spec)
    logits = inputs.moe_logits(spec)
    full = moe.moe_ffn(x, logits, w1, w2, 2, alpha1=0.5, alpha2=2.0)
    pick = [0, 7, 49]
    tok = moe.moe_ffn_tokens(x[pick], logits[pick], lambda e: w1[e], lambda e: w2[e], 2, alpha1=0.5, alpha2=2.0)
    assert np.array_equal(tok["y"], full["y"][pick])
    for i, t in enumerate(pick):
        for j in range(2):
            r = full["inv_perm"][t, j]
            assert np.array_equal(tok["a2_q"][i, j], full["a2_q"][r])
            assert np.array_equal(tok["a2_sf"][i, j], full["a2_sf"][r])
