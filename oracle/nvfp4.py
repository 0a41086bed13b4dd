"""NVFP4 numerics oracle: E4M3 / E2M1 codecs, per-16 block quantiser, SF layout.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``): never imported by the
CUDA library and importing nothing from it.

Sources (the "nvfp4-megamoe-kernel" pages):

* "NVFP4-1.1 Approach, Part 2" -- the FP8 E4M3 cast debugging (bias 7; the
  subnormal step m * 2^-9; exponent 15 is a normal binade except mantissa 7,
  which is NaN, so the largest finite value is 0x7e = 448; a mantissa that rounds
  up to 8 carries into the exponent, so 250 -> 256 = 0x78, not 240 = 0x77), the
  E2M1 nibble rule (half-step hs = RNE(2 * min(|s|, 6)) followed by the
  ``step_to_idx`` table; the worked case s = 5.25 -> hs = 10 -> nibble 6) and the
  per-16 block scale written as one E4M3 byte next to 8 packed nibble bytes.
* "NVFP4 MegaMoE Debug Log", sections "What the forward mapping does",
  "Source strides", "Allocation" and "CUTLASS SF Layout" -- the K-major SF atom
  Shape<Shape<32,4>, Shape<16,4>> / Stride<Stride<16,4>, Stride<0,1>> tiled over
  (M|N, K, L) with Step<2,1,3>, and its inverse mn = f0 + 32 f1 + 128 f2,
  k_sf = f4 + 4 f5.

Readings where the pages are silent (each listed in the design notes):

* the block scale is amax / 6 in fp32 (IEEE round-to-nearest), global scale 1;
* values are divided by the *decoded* E4M3 scale, fp32 IEEE division;
* a zero scale (amax/6 rounds to E4M3 zero) gives magnitude index 0 for every
  element, with the sign bit still taken from the value;
* nibble sign = signbit(v) (so -0.1 with a large scale encodes as 0x8);
* element 2i of a block goes to the low nibble of byte i.

All floating-point decisions that produce an integer code are taken in fp32,
the precision the GPU kernels use.
"""
from __future__ import annotations

import math

import numpy as np

# ---------------------------------------------------------------- FP8 E4M3 --
E4M3_BIAS = 7
E4M3_MAX_CODE = 0x7E        # 448.0, the largest finite magnitude
E4M3_NAN_CODE = 0x7F        # exponent 15, mantissa 7


def e4m3_decode(code: int) -> float:
    """Value of one FP8 E4M3 byte (Approach Part 2, FP8 cast section).

    sign = bit 7, e = bits 6..3, m = bits 2..0.  e == 0: m * 2^-9 (subnormal,
    i.e. 2^(1-7) * m/8).  e > 0: 2^(e-7) * (1 + m/8).  e == 15 and m == 7: NaN.
    There is no infinity.
    """
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 15 and m == 7:
        return math.nan
    if e == 0:
        mag = m * 2.0 ** -9
    else:
        mag = 2.0 ** (e - E4M3_BIAS) * (1.0 + m / 8.0)
    return sign * mag


# the 127 finite non-negative values, indexed by code 0x00..0x7E
_E4M3_POS = np.array([e4m3_decode(c) for c in range(E4M3_MAX_CODE + 1)], dtype=np.float64)
# decode table for all 256 codes as fp32 (exact: every E4M3 value is an fp32 value)
E4M3_TABLE_F32 = np.array([e4m3_decode(c) for c in range(256)], dtype=np.float32)


def e4m3_encode(x: float) -> int:
    """Round a non-negative value to the nearest finite E4M3 code (scalar, brute force).

    Nearest of the 127 finite non-negative codes in exact (float64) distance,
    ties to the even code (= even mantissa, which is round-to-nearest-even), and
    anything above 448 saturates to 0x7E -- the NaN code 0x7F is never returned.
    This is the textbook definition the pages' hand-written cast converges to
    (mantissa carry 250 -> 0x78, clamp at 448, NaN guard).
    """
    if not x >= 0.0:
        raise ValueError("block scales are non-negative and finite")
    best_code, best_dist = 0, math.inf
    for code in range(E4M3_MAX_CODE + 1):
        d = abs(float(_E4M3_POS[code]) - x)
        if d < best_dist or (d == best_dist and code % 2 == 0):
            best_code, best_dist = code, d
    return best_code


def e4m3_encode_array(x: np.ndarray) -> np.ndarray:
    """Vectorised ``e4m3_encode`` (same rule; checked against the scalar form)."""
    x = np.asarray(x, dtype=np.float64)
    if np.any(~(x >= 0.0)):
        raise ValueError("block scales are non-negative and finite")
    hi = np.searchsorted(_E4M3_POS, x, side="left")          # first value >= x
    hi = np.minimum(hi, E4M3_MAX_CODE)
    lo = np.maximum(hi - 1, 0)
    d_hi = np.abs(_E4M3_POS[hi] - x)
    d_lo = np.abs(x - _E4M3_POS[lo])
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(x >= _E4M3_POS[E4M3_MAX_CODE], E4M3_MAX_CODE, code)
    return code.astype(np.uint8)


# ---------------------------------------------------------------- FP4 E2M1 --
def e2m1_decode_magnitude(idx: int) -> float:
    """Magnitude of a 3-bit E2M1 index (1 exponent bias, 2 exponent bits, 1 mantissa bit).

    e = idx >> 1, m = idx & 1.  e == 0: m * 0.5 (subnormal); else 2^(e-1) * (1 + m/2).
    """
    idx = int(idx)
    e, m = idx >> 1, idx & 1
    if e == 0:
        return m * 0.5
    return 2.0 ** (e - 1) * (1.0 + m / 2.0)


E2M1_MAGNITUDES = tuple(e2m1_decode_magnitude(i) for i in range(8))   # 0 .5 1 1.5 2 3 4 6


def e2m1_decode(nibble: int) -> float:
    """Signed value of a 4-bit E2M1 code (bit 3 = sign)."""
    mag = E2M1_MAGNITUDES[nibble & 7]
    return -mag if nibble & 8 else mag


def _nearest_e2m1_index(t: float) -> int:
    """Nearest E2M1 magnitude index to t in [0, 6]; ties go to the even index (even mantissa)."""
    best, best_d = 0, math.inf
    for i, v in enumerate(E2M1_MAGNITUDES):
        d = abs(v - t)
        if d < best_d or (d == best_d and i % 2 == 0):
            best, best_d = i, d
    return best


def step_to_idx() -> tuple:
    """The half-step table of Approach Part 2: hs (0..12) -> E2M1 magnitude index.

    hs / 2 is the scaled magnitude already rounded to a multiple of 0.5; the
    table maps it to the nearest E2M1 magnitude with ties to the even index.
    The pages pin hs=10 -> 6 and hs=11 -> 7; ties-to-even is the only simple
    rule consistent with hs=10 -> 6 (ties-away would give 7), and it fixes the
    unprinted tie entries hs=5 -> 4 and hs=7 -> 6.
    """
    return tuple(_nearest_e2m1_index(hs / 2.0) for hs in range(13))


STEP_TO_IDX = step_to_idx()
_STEP_TO_IDX_NP = np.array(STEP_TO_IDX, dtype=np.uint8)


def half_step(s: np.float32) -> int:
    """hs = RNE(2 * min(|s|, 6)) (Python's round() is round-half-even, as the pages note)."""
    t = 2.0 * min(abs(float(s)), 6.0)     # exact: s is fp32, the product fits float64
    return int(round(t))


# ------------------------------------------------------- block quantiser --
BLOCK = 16


def quantize_block(v) -> tuple:
    """Quantise 16 fp32 values -> (8 packed bytes, 1 E4M3 scale byte).  Scalar form.

    Steps (Approach Part 2): amax -> bsf = amax / 6 (fp32) -> E4M3 byte ->
    s = v / dec(sf) (fp32) -> hs = RNE(2 min(|s|, 6)) -> step_to_idx -> sign bit ->
    pack element 2i into the low nibble of byte i.
    """
    v = [np.float32(x) for x in v]
    if len(v) != BLOCK:
        raise ValueError("a block holds 16 values")
    amax = max(abs(x) for x in v)
    bsf = np.float32(amax) / np.float32(6.0)
    sf = e4m3_encode(float(bsf))
    d = np.float32(e4m3_decode(sf))
    nibbles = []
    for x in v:
        sign = 1 if np.signbit(x) else 0
        if d == 0:
            idx = 0
        else:
            s = np.float32(x / d)          # fp32 / fp32 -> IEEE fp32 quotient
            idx = STEP_TO_IDX[half_step(s)]
        nibbles.append((sign << 3) | idx)
    packed = bytes(nibbles[2 * i] | (nibbles[2 * i + 1] << 4) for i in range(BLOCK // 2))
    return packed, sf


# Two-level scale (the pages' pipeline carries a per-tensor fp32 global scale
# next to the per-16 E4M3 scales -- "NVFP4 MegaMoE Debug Log", "NVFP4 MoE
# Pipeline": stage_activation returns an input_global_scale and each GEMM's alpha
# is input global scale x weight global scale; the pages print no formula).
# Reading taken here: an encode scale g multiplies the tensor before the per-16
# quantisation, chosen so the tensor's amax lands on the top of the E4M3 x E2M1
# range (6 * 448); dequantisation divides by g.
GLOBAL_RANGE = np.float32(6.0 * 448.0)


def global_scale(x: np.ndarray) -> np.float32:
    """g = fp32(2688 / amax(|x|)); 1 when amax is 0 or the quotient is not finite."""
    x = np.asarray(x, dtype=np.float32)
    amax = np.float32(np.max(np.abs(x))) if x.size else np.float32(0.0)
    if amax == 0:
        return np.float32(1.0)
    with np.errstate(over="ignore", divide="ignore"):
        g = np.float32(GLOBAL_RANGE / amax)
    return g if np.isfinite(g) else np.float32(1.0)


def quantize_rows(x: np.ndarray, gscale=None) -> tuple:
    """Vectorised per-16 quantiser over the last axis.

    x: fp32 [rows, cols] (cols % 16 == 0).  Returns (q uint8 [rows, cols/2],
    sf uint8 [rows, cols/16]) with the SF in plain row-major order.  With an
    encode scale ``gscale`` (two-level scheme) the quantised values are
    fp32(x * gscale), rounded once.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    if gscale is not None:
        x = (x * np.float32(gscale)).astype(np.float32)
    rows, cols = x.shape
    if cols % BLOCK:
        raise ValueError("cols must be a multiple of 16")
    blocks = x.reshape(rows, cols // BLOCK, BLOCK)
    amax = np.max(np.abs(blocks), axis=2)
    bsf = (amax / np.float32(6.0)).astype(np.float32)
    sf = e4m3_encode_array(bsf)
    d = E4M3_TABLE_F32[sf][:, :, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        s = (blocks / d).astype(np.float32)
    t = 2.0 * np.minimum(np.abs(s.astype(np.float64)), 6.0)
    hs = np.rint(t)                                   # round-half-even
    hs = np.where(d == 0, 0.0, hs).astype(np.int64)
    idx = _STEP_TO_IDX_NP[hs]
    nib = (np.signbit(blocks).astype(np.uint8) << 3) | idx
    nib = nib.reshape(rows, cols)
    q = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    return q, sf


def dequantize_rows(q: np.ndarray, sf: np.ndarray, gscale=None) -> np.ndarray:
    """float64 [rows, 2*q.shape[1]] from packed nibbles and row-major SF bytes
    (divided by the encode scale ``gscale`` of the two-level scheme, if given)."""
    q = np.asarray(q, dtype=np.uint8)
    rows, half = q.shape
    nib = np.empty((rows, 2 * half), dtype=np.uint8)
    nib[:, 0::2] = q & 0xF
    nib[:, 1::2] = q >> 4
    table = np.array([e2m1_decode(n) for n in range(16)], dtype=np.float64)
    vals = table[nib]
    scale = E4M3_TABLE_F32[np.asarray(sf, dtype=np.uint8)].astype(np.float64)
    out = vals * np.repeat(scale, BLOCK, axis=1)
    return out if gscale is None else out / np.float64(np.float32(gscale))


def unpack_nibbles(q: np.ndarray) -> np.ndarray:
    """uint8 [rows, 2*cols] nibble codes from packed bytes (low nibble first)."""
    q = np.asarray(q, dtype=np.uint8)
    nib = np.empty(q.shape[:-1] + (2 * q.shape[-1],), dtype=np.uint8)
    nib[..., 0::2] = q & 0xF
    nib[..., 1::2] = q >> 4
    return nib


# ------------------------------------------------------- swizzled SF layout --
SF_ATOM_MN = 128      # rows covered by one 512-byte atom
SF_ATOM_KSF = 4       # scale columns (= 64 K elements) covered by one atom
SF_ATOM_BYTES = 512


def sf_padded_bytes(mn: int, k_elems: int) -> int:
    """size(filter_zeros(layout)) of the swizzled SF for an mn x k matrix
    (Debug Log, "Allocation"): ceil(mn/128) * ceil(k/64) * 512 bytes."""
    return -(-mn // SF_ATOM_MN) * -(-k_elems // (BLOCK * SF_ATOM_KSF)) * SF_ATOM_BYTES


def sf_offset(mn: int, k_sf: int, k_sf_total: int) -> int:
    """Byte offset of scale (mn, k_sf) in the swizzled layout (closed form).

    Read off the atom of the Debug Log's "CUTLASS SF Layout": mode 0 (32,4):(16,4)
    covers M|N, mode 1 (16,4):(0,1) covers K, atoms tiled with K innermost
    (Step<2,1,3>).
    """
    k4 = -(-k_sf_total // SF_ATOM_KSF)
    atom = (mn // SF_ATOM_MN) * k4 + k_sf // SF_ATOM_KSF
    return atom * SF_ATOM_BYTES + (mn % 32) * 16 + ((mn // 32) % 4) * 4 + (k_sf % 4)


def swizzle_sf(sf_lin: np.ndarray) -> np.ndarray:
    """Row-major SF bytes [mn, k_sf] -> padded swizzled buffer (padding bytes are 0)."""
    sf_lin = np.asarray(sf_lin, dtype=np.uint8)
    mn, k_sf = sf_lin.shape
    out = np.zeros(sf_padded_bytes(mn, k_sf * BLOCK), dtype=np.uint8)
    for m in range(mn):
        for k in range(k_sf):
            out[sf_offset(m, k, k_sf)] = sf_lin[m, k]
    return out


def swizzle_sf_fast(sf_lin: np.ndarray) -> np.ndarray:
    """Vectorised ``swizzle_sf`` (checked against the loop form)."""
    sf_lin = np.asarray(sf_lin, dtype=np.uint8)
    mn, k_sf = sf_lin.shape
    out = np.zeros(sf_padded_bytes(mn, k_sf * BLOCK), dtype=np.uint8)
    m = np.arange(mn)[:, None]
    k = np.arange(k_sf)[None, :]
    k4 = -(-k_sf // SF_ATOM_KSF)
    off = ((m // 128) * k4 + k // 4) * 512 + (m % 32) * 16 + ((m // 32) % 4) * 4 + (k % 4)
    out[off.ravel()] = sf_lin.ravel()
    return out


def unswizzle_sf(sf_swz: np.ndarray, mn: int, k_sf: int) -> np.ndarray:
    """Inverse of ``swizzle_sf_fast`` on the valid region."""
    sf_swz = np.asarray(sf_swz, dtype=np.uint8)
    m = np.arange(mn)[:, None]
    k = np.arange(k_sf)[None, :]
    k4 = -(-k_sf // SF_ATOM_KSF)
    off = ((m // 128) * k4 + k // 4) * 512 + (m % 32) * 16 + ((m // 32) % 4) * 4 + (k % 4)
    return sf_swz[off]


# ------------------------------------------------------- SwiGLU quantiser --
def deinterleave_gu8(gu: np.ndarray) -> tuple:
    """Split columns interleaved at granularity 8 ([g0(8) u0(8) g1(8) u1(8) ...])
    into (gate, up) (Approach Part 2, interleave_l1_weights / activation view)."""
    gu = np.asarray(gu)
    rows, cols2 = gu.shape
    if cols2 % 16:
        raise ValueError("interleaved width must be a multiple of 16")
    v = gu.reshape(rows, cols2 // 16, 2, 8)
    return v[:, :, 0, :].reshape(rows, cols2 // 2), v[:, :, 1, :].reshape(rows, cols2 // 2)


def silu64(g: np.ndarray) -> np.ndarray:
    """silu(g) = g / (1 + exp(-g)) in float64."""
    g = np.asarray(g, dtype=np.float64)
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


def swiglu_h(gate: np.ndarray, up: np.ndarray) -> np.ndarray:
    """h = silu(g) * u evaluated in float64, then rounded once to fp32 (the
    precision the quantiser works in)."""
    return (silu64(gate) * np.asarray(up, dtype=np.float64)).astype(np.float32)


def quantize_deinterleave_gu8(gu: np.ndarray, gscale=None) -> tuple:
    """The pages' deinterleave + quantise (Approach Part 2, K2 as they run it): from
    columns interleaved at granularity 8, keep the second 8 of every 16 (the up /
    already-SwiGLU'd slots) and quantise them per 16 -> (q, sf_row_major, kept values)."""
    _, up = deinterleave_gu8(gu)
    kept = np.asarray(up, dtype=np.float32)
    q, sf = quantize_rows(kept, gscale)
    return q, sf, kept


def quantize_swiglu_gu8(gu: np.ndarray, gscale=None) -> tuple:
    """The standalone SwiGLU + NVFP4 quantiser: interleaved gate/up -> (q, sf_row_major, h).
    h is returned unscaled; an encode scale applies to the quantised values only."""
    g, u = deinterleave_gu8(gu)
    h = swiglu_h(g, u)
    q, sf = quantize_rows(h, gscale)
    return q, sf, h
