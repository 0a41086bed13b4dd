"""Pins for the oracle's FP8 E4M3 and FP4 E2M1 codecs (CPU only).

Each check ties the oracle to something other than itself: values printed on
"NVFP4-1.1 Approach, Part 2" (tests/golden/), PyTorch's float8_e4m3fn cast (the
library routine those pages validated against), PyTorch's reference rounding to
E2M1 (for the half-step table), structural facts of the formats, and
hand-derived cases.
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle import nvfp4

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                yield line.split()


# ----------------------------------------------------------------- E4M3 --
def test_e4m3_golden_values_from_pages():
    n = 0
    for kind, inp, exp, *_ in _rows("e4m3_pages.txt"):
        if kind == "decode":
            got = nvfp4.e4m3_decode(int(inp, 16))
            if exp == "nan":
                assert math.isnan(got)
            else:                                     # the page prints 6 decimals
                assert abs(got - float(exp)) <= 5e-7 * max(1.0, float(exp)), (inp, got)
        else:
            assert nvfp4.e4m3_encode(float(inp)) == int(exp, 16), (inp, exp)
        n += 1
    assert n == 9


def test_e4m3_bias_is_7():
    # 1.0 is exponent field 7, mantissa 0 -> code 0x38 (bias 7, not 8)
    assert nvfp4.e4m3_decode(0x38) == 1.0
    assert nvfp4.e4m3_encode(1.0) == 0x38


def test_e4m3_decode_matches_torch_all_256_codes():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).float().numpy()
    for c in range(256):
        got = nvfp4.e4m3_decode(c)
        if math.isnan(ref[c]):
            assert math.isnan(got), hex(c)
        else:
            assert got == ref[c], (hex(c), got, ref[c])
    # exactly two NaN codes, no infinity
    assert sum(math.isnan(nvfp4.e4m3_decode(c)) for c in range(256)) == 2


def test_e4m3_structure():
    pos = [nvfp4.e4m3_decode(c) for c in range(0x7F)]
    assert all(a < b for a, b in zip(pos, pos[1:]))          # strictly increasing
    assert pos[1] == 2.0 ** -9 and pos[-1] == 448.0
    # subnormal step equals the step of the first normal binade (continuity)
    assert pos[8] - pos[7] == pos[1] - pos[0] == pos[9] - pos[8]
    # each normal binade holds 8 equally spaced values
    for e in range(1, 16):
        vals = [nvfp4.e4m3_decode((e << 3) | m) for m in range(8 if e < 15 else 7)]
        steps = {b - a for a, b in zip(vals, vals[1:])}
        assert steps == {2.0 ** (e - 10)}
    # negative codes mirror positive ones
    for c in range(0x7F):
        assert nvfp4.e4m3_decode(c | 0x80) == -nvfp4.e4m3_decode(c)


def _torch_encode(x):
    t = torch.tensor(np.asarray(x, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_encode_matches_torch_on_ties_and_random():
    pos = np.array([nvfp4.e4m3_decode(c) for c in range(0x7F)])
    mids = (pos[:-1] + pos[1:]) / 2                 # every exact tie (exact in fp32)
    eps = np.float32(1.0) + np.float32(2.0 ** -20)
    rng = np.random.default_rng(11)
    xs = np.concatenate([pos, mids, mids * eps, mids / eps,
                         rng.uniform(0, 460, 4000), np.exp(rng.uniform(-14, 6, 4000))])
    xs = xs.astype(np.float32)
    xs = xs[xs < 464]                                # torch returns NaN from 464 up
    ref = _torch_encode(xs)
    got = nvfp4.e4m3_encode_array(xs.astype(np.float64))
    assert np.array_equal(got, ref)
    for x in xs[::37]:
        assert nvfp4.e4m3_encode(float(x)) == _torch_encode([x])[0]


def test_e4m3_encode_saturates_instead_of_nan():
    for x in (448.0, 455.0, 464.0, 470.0, 1e4, 3.0e38):
        assert nvfp4.e4m3_encode(x) == 0x7E
    assert np.all(nvfp4.e4m3_encode_array(np.array([464.0, 1e6])) == 0x7E)


def test_e4m3_encode_decode_roundtrip_all_finite_codes():
    for c in range(0x7F):
        assert nvfp4.e4m3_encode(nvfp4.e4m3_decode(c)) == c
    # the two zeros: -0 re-encodes as +0 (scales are magnitudes)
    assert nvfp4.e4m3_encode(abs(nvfp4.e4m3_decode(0x80))) == 0x00


def test_e4m3_vector_matches_scalar():
    rng = np.random.default_rng(5)
    xs = np.concatenate([np.exp(rng.uniform(-16, 7, 3000)), [0.0, 2.0 ** -10, 2.0 ** -9]])
    got = nvfp4.e4m3_encode_array(xs)
    for x, g in zip(xs, got):
        assert nvfp4.e4m3_encode(float(x)) == g


def test_e4m3_zero_scale_boundary():
    # half the smallest subnormal ties to the even code 0x00; just above goes to 0x01
    assert nvfp4.e4m3_encode(2.0 ** -10) == 0x00
    assert nvfp4.e4m3_encode(2.0 ** -10 * (1 + 2 ** -20)) == 0x01
    # subnormal / normal boundary: 7.5 * 2^-9 ties to 0x08 (even)
    assert nvfp4.e4m3_encode(7.5 * 2.0 ** -9) == 0x08


# ----------------------------------------------------------------- E2M1 --
def test_e2m1_grid():
    # 1 mantissa bit, 2 exponent bits, bias 1: the half-step grid of the pages
    # (steps of 0.5 near zero, clamp at 6)
    assert nvfp4.E2M1_MAGNITUDES == (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)
    assert max(nvfp4.E2M1_MAGNITUDES) == 6.0
    for n in range(16):
        v = nvfp4.e2m1_decode(n)
        assert math.copysign(1.0, v) == (-1.0 if n & 8 else 1.0)
        assert abs(v) == nvfp4.E2M1_MAGNITUDES[n & 7]


def test_e2m1_golden_from_pages():
    seen = 0
    for kind, inp, exp in _rows("e2m1_pages.txt"):
        if kind == "step":
            assert nvfp4.STEP_TO_IDX[int(inp)] == int(exp)
        elif kind == "halfstep":
            assert nvfp4.half_step(np.float32(float(inp))) == int(exp)
        elif kind == "scaled":
            assert nvfp4.STEP_TO_IDX[nvfp4.half_step(np.float32(float(inp)))] == int(exp)
        seen += 1
    assert seen == 4


def _torch_e2m1_rne():
    """PyTorch's reference rounding of fp32 to a small float format (round to
    nearest, ties to even, saturating at the largest finite value), from its
    microscaling test utilities -- written independently of this oracle; None
    where that module cannot be imported.  Importing it pulls in PyTorch's
    test-suite base, which wants the ``expecttest`` package; where that is
    absent an empty stand-in satisfies the import (nothing of it is used)."""
    import sys
    import types
    import unittest
    stub = None
    if "expecttest" not in sys.modules:
        try:
            import expecttest  # noqa: F401
        except ImportError:
            stub = types.ModuleType("expecttest")
            stub.TestCase = unittest.TestCase
            sys.modules["expecttest"] = stub
    try:
        from torch.testing._internal.common_quantized import _f32_to_floatx_unpacked
    except Exception:
        return None
    finally:
        if stub is not None and sys.modules.get("expecttest") is stub:
            del sys.modules["expecttest"]
    return lambda vals: _f32_to_floatx_unpacked(torch.tensor(vals, dtype=torch.float32), 2, 1).tolist()


def test_step_table_is_rne_onto_the_e2m1_grid():
    """The second stage of the pages' rule maps the half-step value hs/2 onto
    the E2M1 grid.  The pages print hs = 10 -> 6 and hs = 11 -> 7; reading the
    table as round-to-nearest-even onto the grid (the only simple rule that
    gives hs = 10 -> 6), every entry -- including the unprinted ties hs = 5
    (2.5 -> 2) and hs = 7 (3.5 -> 4) -- must equal PyTorch's independent
    E2M1 rounding of hs/2."""
    rne = _torch_e2m1_rne()
    if rne is None:
        pytest.skip("PyTorch's small-float reference rounding is not importable")
    codes = rne([hs / 2.0 for hs in range(13)])
    assert tuple(codes) == nvfp4.STEP_TO_IDX
    # the same routine applied to the unrounded 5.25 gives the direct-RNE code 7,
    # which the pages' two-stage rule does not (it pre-rounds to half steps)
    assert rne([5.25]) == [7] and nvfp4.STEP_TO_IDX[nvfp4.half_step(np.float32(5.25))] == 6


# hand-derived: scaled magnitude -> half step (round-half-even of 2s) -> index
HAND_TABLE = {
    0.0: 0, 0.2: 0, 0.25: 0, 0.26: 1, 0.5: 1, 0.75: 2, 1.0: 2, 1.25: 2, 1.5: 3,
    1.75: 4, 2.0: 4, 2.25: 4, 2.5: 4, 2.75: 5, 3.0: 5, 3.25: 5, 3.5: 6, 3.75: 6,
    4.0: 6, 4.25: 6, 4.75: 6, 5.0: 6, 5.25: 6, 5.5: 7, 5.75: 7, 6.0: 7, 9.0: 7,
}


def test_two_stage_rule_hand_table():
    for s, idx in HAND_TABLE.items():
        assert nvfp4.STEP_TO_IDX[nvfp4.half_step(np.float32(s))] == idx, s


def test_two_stage_rule_differs_from_direct_rne_only_where_expected():
    # direct RNE onto the E2M1 grid maps 5.25 to 6.0 (index 7): the pages' rule
    # deliberately does not (it pre-rounds to half steps first).
    assert nvfp4._nearest_e2m1_index(5.25) == 7
    assert nvfp4.STEP_TO_IDX[nvfp4.half_step(np.float32(5.25))] == 6
