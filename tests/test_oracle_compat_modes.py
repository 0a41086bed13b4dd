"""Pins of the oracle's two compatibility paths from the pages' CuTeDSL era:
the deinterleave + quantise mode (keep the second 8 of every 16 interleaved
columns, quantise them) and the compact BF16 SwiGLU output.

* the deinterleave mode on an interleaved buffer whose kept slots hold a matrix
  M equals the plain quantisation of M (closed form), whatever the other slots
  hold;
* the compact output rounds once: it equals BF16 of the fp32 h the fused
  NVFP4 epilogue quantises, and for gate values large enough that silu(g) == g
  in fp32 it is bf16(g * u).
"""
import numpy as np

from oracle import moe as omoe
from oracle import nvfp4 as onv


def _interleave(gate, up):
    rows, n = gate.shape
    out = np.empty((rows, n // 8, 2, 8), dtype=np.float32)
    out[:, :, 0, :] = gate.reshape(rows, n // 8, 8)
    out[:, :, 1, :] = up.reshape(rows, n // 8, 8)
    return out.reshape(rows, 2 * n)


def test_deinterleave_mode_is_plain_quantisation_of_the_kept_slots():
    rng = np.random.default_rng(90)
    m = rng.standard_normal((40, 256)).astype(np.float32)
    junk = (rng.standard_normal((40, 256)) * 1e4).astype(np.float32)
    q, sf, kept = onv.quantize_deinterleave_gu8(_interleave(junk, m))
    q0, sf0 = onv.quantize_rows(m)
    assert np.array_equal(kept, m) and np.array_equal(q, q0) and np.array_equal(sf, sf0)


def test_compact_swiglu_output_rounds_once():
    rng = np.random.default_rng(91)
    g_full = rng.standard_normal((16, 512)) * 3
    h_bf16 = omoe.l1_swiglu_bf16(g_full)
    _, _, h = omoe.l1_swiglu_requant(g_full)
    assert np.array_equal(h_bf16, omoe.round_to_bf16(h.astype(np.float64)))
    gate = np.full((4, 64), 120.0)
    up = rng.standard_normal((4, 64))
    out = omoe.l1_swiglu_bf16(_interleave(gate.astype(np.float32), up.astype(np.float32)).astype(np.float64))
    assert np.array_equal(out, omoe.round_to_bf16(np.float32(120.0) * up.astype(np.float32)))
