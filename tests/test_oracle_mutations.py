"""Plant plausible mistakes in the oracle (on the CPU only) and check that the
pins catch each one: a pin that a wrong oracle also passes pins nothing."""
import math

import numpy as np
import pytest

from oracle import moe, nvfp4

import test_oracle_codecs as codecs
import test_oracle_moe as moe_tests
import test_oracle_quant as quant


def _decode_bias8(code):
    code = int(code) & 0xFF
    e, m = (code >> 3) & 0xF, code & 7
    if e == 15 and m == 7:
        return math.nan
    mag = m * 2.0 ** -10 if e == 0 else 2.0 ** (e - 8) * (1 + m / 8)
    return -mag if code & 0x80 else mag


def _encode_truncating(x):
    # mantissa rounding without the carry into the exponent (the 250 -> 240 bug)
    best = 0
    for c in range(0x7F):
        if nvfp4._E4M3_POS[c] <= x:
            best = c
    return best


def _ties_away_table():
    # hs = 5, 7, 10 (the E2M1-grid ties) rounded away from zero
    return (0, 1, 2, 3, 4, 5, 5, 6, 6, 6, 7, 7, 7)


def _hs5_up_table():
    # only the unprinted tie hs = 5 (2.5) rounded up to 3
    return (0, 1, 2, 3, 4, 5, 5, 6, 6, 6, 6, 7, 7)


def _half_up(s):
    return int(math.floor(2.0 * min(abs(float(s)), 6.0) + 0.5))


def _offset_m_inner(mn, k_sf, k_sf_total):
    # atom tiling with M atoms innermost instead of K (Step order swapped)
    m_atoms = 1 << 20
    atom = (k_sf // 4) * m_atoms + mn // 128
    return atom * 512 + (mn % 32) * 16 + ((mn // 32) % 4) * 4 + (k_sf % 4)


def _dequant_high_first(q, sf):
    q = np.asarray(q, np.uint8)
    swapped = ((q & 0xF) << 4) | (q >> 4)
    return ORIG_DEQUANT(swapped, sf)


ORIG_DEQUANT = nvfp4.dequantize_rows


def _route_ties_high(logits, k):
    logits = np.asarray(logits, np.float32)
    order = np.argsort(-logits[:, ::-1].astype(np.float64), axis=1, kind="stable")[:, :k]
    order = logits.shape[1] - 1 - order
    sel = np.take_along_axis(logits, order, 1).astype(np.float64)
    z = np.exp(sel - sel[:, :1])
    return order.astype(np.int32), z / z.sum(1, keepdims=True)


MUTATIONS = [
    ("e4m3 bias 8", "e4m3_decode", _decode_bias8, codecs.test_e4m3_golden_values_from_pages),
    ("e4m3 truncating encode", "e4m3_encode", _encode_truncating, codecs.test_e4m3_golden_values_from_pages),
    ("step table ties away", "STEP_TO_IDX", _ties_away_table(), codecs.test_e2m1_golden_from_pages),
    ("step table hs=5 up", "STEP_TO_IDX", _hs5_up_table(), codecs.test_step_table_is_rne_onto_the_e2m1_grid),
    ("half-up half step", "half_step", _half_up, codecs.test_e2m1_golden_from_pages),
    ("SF atoms M-innermost", "sf_offset", _offset_m_inner, quant.test_sf_closed_form_equals_cute_atom_tiling),
    ("nibble order high-first", "dequantize_rows", _dequant_high_first,
     moe_tests.test_dequantize_matches_scalar_decoders_and_nibble_order),
]


@pytest.mark.parametrize("name,attr,value,check", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_oracle_mistake(monkeypatch, name, attr, value, check):
    check()                                       # passes on the real oracle
    monkeypatch.setattr(nvfp4, attr, value)
    with pytest.raises(AssertionError):
        check()


def test_pins_catch_routing_tie_break_mistake(monkeypatch):
    moe_tests.test_route_topk_brute_force()
    monkeypatch.setattr(moe, "route_topk", _route_ties_high)
    with pytest.raises(AssertionError):
        moe_tests.test_route_topk_brute_force()
