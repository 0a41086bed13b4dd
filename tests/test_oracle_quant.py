"""Pins for the oracle's per-16 block quantiser, SwiGLU and SF layout (CPU only)."""
import numpy as np
import pytest
import scipy.special

import inputs
from oracle import nvfp4

from test_oracle_codecs import HAND_TABLE


def _scalar_rows(x):
    rows, cols = x.shape
    q = np.zeros((rows, cols // 2), np.uint8)
    sf = np.zeros((rows, cols // 16), np.uint8)
    for r in range(rows):
        for b in range(cols // 16):
            p, s = nvfp4.quantize_block(x[r, 16 * b:16 * b + 16])
            q[r, 8 * b:8 * b + 8] = np.frombuffer(p, np.uint8)
            sf[r, b] = s
    return q, sf


def test_vector_quantiser_matches_scalar_form():
    x = inputs.plain_input_with_ties(3, 24, 256)
    x[0, :16] = 0.0                                     # all-zero block
    x[1, :16] = -0.0
    x[2, 16:32] = np.float32(1e-30)                     # zero scale, tiny values
    x[3, 32:48] *= np.float32(1e6)                      # saturated scale
    q, sf = nvfp4.quantize_rows(x)
    q2, sf2 = _scalar_rows(x)
    assert np.array_equal(q, q2) and np.array_equal(sf, sf2)


def test_planted_ties_follow_hand_table():
    # one element 6 * 2^q fixes the scale at exactly 2^q; the others are m * 2^q
    ms = [m for m in HAND_TABLE if m <= 6.0 and float(np.float32(m)) == m]
    for q in (-9, -7, -6, 0, 3, 8):
        for i in range(0, len(ms), 15):
            chunk = (ms[i:i + 15] + [0.0] * 15)[:15]
            vals = np.array([6.0] + chunk, np.float32) * np.float32(2.0 ** q)
            p, sfb = nvfp4.quantize_block(vals)
            assert nvfp4.e4m3_decode(sfb) == 2.0 ** q
            nib = nvfp4.unpack_nibbles(np.frombuffer(p, np.uint8)[None])[0]
            for v, n in zip(vals, nib):
                assert n == HAND_TABLE[float(v) / 2.0 ** q], (q, v, n)


def test_sign_bits_and_zero_scale():
    vals = np.array([-1e-30, 1e-30, -0.0, 0.0] + [0.0] * 12, np.float32)
    p, sfb = nvfp4.quantize_block(vals)
    assert sfb == 0
    nib = nvfp4.unpack_nibbles(np.frombuffer(p, np.uint8)[None])[0]
    assert list(nib[:4]) == [8, 0, 8, 0]
    # -0.1 next to a large value: magnitude rounds to 0 but the sign bit stays
    vals = np.zeros(16, np.float32)
    vals[0], vals[1] = 6.0, -0.1
    p, _ = nvfp4.quantize_block(vals)
    nib = nvfp4.unpack_nibbles(np.frombuffer(p, np.uint8)[None])[0]
    assert nib[0] == 7 and nib[1] == 8


def test_scale_is_e4m3_of_amax_over_6():
    rng = np.random.default_rng(2)
    x = (rng.standard_normal((64, 64)) * np.exp(rng.uniform(-9, 9, (64, 1)))).astype(np.float32)
    _, sf = nvfp4.quantize_rows(x)
    amax = np.abs(x.reshape(64, 4, 16)).max(axis=2)
    for a, s in zip(amax.ravel(), sf.ravel()):
        # fp32 division by 6, then the E4M3 nearest (checked against torch's cast
        # below 464, saturation above)
        bsf = np.float32(a) / np.float32(6)
        assert s == nvfp4.e4m3_encode(float(bsf))


def test_dequant_error_bound():
    rng = np.random.default_rng(4)
    x = rng.standard_t(3, (128, 256)).astype(np.float32)
    q, sf = nvfp4.quantize_rows(x)
    dq = nvfp4.dequantize_rows(q, sf)
    d = np.repeat(nvfp4.E4M3_TABLE_F32[sf].astype(np.float64), 16, axis=1)
    s = np.abs(x / d)
    # half-step rounding (<= 0.25) plus snapping to the E2M1 grid (half spacing)
    bound = 0.25 + np.where(s < 2, 0.0, np.where(s < 4, 0.5, 1.0)) + np.maximum(s - 6, 0)
    assert np.all(np.abs(dq / d - x / d) <= bound + 1e-6)
    assert np.all(np.sign(dq) * np.sign(x) >= 0)


def test_swiglu_matches_scipy_and_pages_deinterleave_view():
    rng = np.random.default_rng(8)
    gu = rng.standard_normal((5, 96)).astype(np.float32)
    g, u = nvfp4.deinterleave_gu8(gu)
    # the pages' activation view: reshape(T, -1, 16)[:, :, 8:] picks the up half
    assert np.array_equal(u, gu.reshape(5, -1, 16)[:, :, 8:].reshape(5, -1))
    assert np.array_equal(g, gu.reshape(5, -1, 16)[:, :, :8].reshape(5, -1))
    h = nvfp4.swiglu_h(g, u)
    ref = (g.astype(np.float64) * scipy.special.expit(g.astype(np.float64)) * u).astype(np.float32)
    assert np.array_equal(h, ref)
    assert nvfp4.silu64(np.array([0.0]))[0] == 0.0
    assert np.float32(nvfp4.silu64(np.array([64.0]))[0]) == np.float32(64.0)


def test_planted_gu8_blocks_are_exact_ties():
    t, plant = inputs.quantizer_input(dict(seed=9), rows=64, cols=256)
    gu = t.float().numpy()
    q, sf, h = nvfp4.quantize_swiglu_gu8(gu)
    nb = 256 // 16
    for blk in plant["midpoint"]:
        r, b = divmod(int(blk), nb)
        hb = h[r, 16 * b:16 * b + 16]
        d = nvfp4.e4m3_decode(sf[r, b])
        assert np.max(np.abs(hb)) == 6 * d
        for v, n in zip(hb, nvfp4.unpack_nibbles(q[r:r + 1, 8 * b:8 * b + 8])[0]):
            assert (n & 7) == HAND_TABLE[abs(float(v)) / d]
    for blk in plant["saturate"]:
        r, b = divmod(int(blk), nb)
        if np.max(np.abs(h[r, 16 * b:16 * b + 16])) / 6 > 464:
            assert sf[r, b] == 0x7E


# ------------------------------------------------------------- SF layout --
def _cute_eval(shape, stride, coord):
    """Evaluate a nested CuTe layout at a nested coordinate (inner product)."""
    if isinstance(shape, tuple):
        return sum(_cute_eval(s, d, c) for s, d, c in zip(shape, stride, coord))
    assert 0 <= coord < shape
    return coord * stride


def _cute_split(x, shape):
    """Colexicographic split of a flat index into a (possibly nested) shape."""
    if isinstance(shape, tuple):
        out = []
        for s in shape:
            size = int(np.prod(_flat(s)))
            out.append(_cute_split(x % size, s))
            x //= size
        return tuple(out)
    return x


def _flat(s):
    return sum((_flat(t) for t in s), []) if isinstance(s, tuple) else [s]


def test_sf_closed_form_equals_cute_atom_tiling():
    # atom: Shape<Shape<32,4>, Shape<16,4>> Stride<Stride<16,4>, Stride<0,1>> (512 B),
    # tiled over (MN, K) with K atoms innermost (Step<2,1,3>)
    atom_shape = ((32, 4), (16, 4))
    atom_stride = ((16, 4), (0, 1))
    for mn_total, k_total in ((128, 64), (256, 192), (384, 512), (200, 80)):
        k_atoms = -(-k_total // 64)
        for mn in range(0, -(-mn_total // 128) * 128, 7):
            for k in range(0, k_atoms * 64, 16):
                inner = _cute_eval(atom_shape, atom_stride,
                                   (_cute_split(mn % 128, (32, 4)), _cute_split(k % 64, (16, 4))))
                tile = (mn // 128) * k_atoms + (k // 64)
                assert tile * 512 + inner == nvfp4.sf_offset(mn, k // 16, k_total // 16)


def test_sf_inverse_formula_from_debug_log():
    # mn = f0 + 32 f1 + 128 f2, k_sf = f4 + 4 f5 (f3 is the stride-0 mode)
    k_sf_total = 12
    for off in range(nvfp4.sf_padded_bytes(256, 16 * k_sf_total)):
        atom, inner = divmod(off, 512)
        f2, f5 = divmod(atom, 3)
        f0, rest = divmod(inner, 16)
        f1, f4 = divmod(rest, 4)
        mn, k_sf = f0 + 32 * f1 + 128 * f2, f4 + 4 * f5
        assert nvfp4.sf_offset(mn, k_sf, k_sf_total) == off


@pytest.mark.parametrize("mn,k_sf", [(1, 1), (3, 3), (128, 4), (130, 5), (300, 9), (512, 448 // 16)])
def test_sf_swizzle_is_a_bijection_and_roundtrips(mn, k_sf):
    rng = np.random.default_rng(mn * 31 + k_sf)
    lin = rng.integers(1, 256, (mn, k_sf), dtype=np.uint8)
    swz = nvfp4.swizzle_sf(lin)
    assert np.array_equal(swz, nvfp4.swizzle_sf_fast(lin))
    assert len(swz) == nvfp4.sf_padded_bytes(mn, 16 * k_sf)
    offs = {nvfp4.sf_offset(m, k, k_sf) for m in range(mn) for k in range(k_sf)}
    assert len(offs) == mn * k_sf                     # injective
    assert np.count_nonzero(swz) == mn * k_sf         # padding stays zero
    assert np.array_equal(nvfp4.unswizzle_sf(swz, mn, k_sf), lin)


def test_sf_bands_concatenate():
    # the SF of 128-padded groups, concatenated, is the SF of the stacked matrix
    rng = np.random.default_rng(1)
    a = rng.integers(0, 256, (128, 8), dtype=np.uint8)
    b = rng.integers(0, 256, (256, 8), dtype=np.uint8)
    whole = nvfp4.swizzle_sf_fast(np.concatenate([a, b]))
    assert np.array_equal(whole, np.concatenate([nvfp4.swizzle_sf_fast(a), nvfp4.swizzle_sf_fast(b)]))

