"""GPU parity of the pages' two compatibility paths: the deinterleave + quantise
mode of nvfp4_quantize (keep the second 8 of every 16 interleaved columns) and
the compact BF16 SwiGLU epilogue of nvfp4_grouped_gemm, against the oracle
(``nvfp4.quantize_deinterleave_gu8``, ``moe.l1_swiglu_bf16``).

The quantiser mode is bit-exact (its inputs are the BF16 values themselves).
The compact output is within relative Frobenius 2e-3 of BF16(float64 h) with
nearly every value identical (the fast SiLU moves a few values across a BF16
rounding boundary), equal on both tile kernels, and writes real rows only.
"""
import contextlib

import numpy as np
import pytest
import torch

import inputs
from oracle import moe as omoe
from oracle import nvfp4 as onv

from gpu_util import built_lib, dev, host, rel_frobenius

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    built_lib()
    import nvfp4_block_scaled_moe_gb300 as nv
    return nv


@pytest.mark.parametrize("rows,cols", [(1, 16), (129, 512), (300, 2048)])
def test_deinterleave_mode_bit_exact(nv, rows, cols):
    gu_t, _ = inputs.quantizer_input(dict(seed=rows + 3 * cols), rows=rows, cols=cols)
    q = torch.empty((rows, cols // 2), dtype=torch.uint8, device="cuda")
    sf = torch.empty(nv.sf_bytes(rows, cols), dtype=torch.uint8, device="cuda")
    h = torch.empty((rows, cols), dtype=torch.float32, device="cuda")
    nv.nvfp4_quantize(gu_t.cuda(), cols, nv.MODE_DEINTERLEAVE_GU8, q, sf, h_debug=h)
    nv.nvfp4_device_status()
    oq, osf, kept = onv.quantize_deinterleave_gu8(gu_t.float().numpy())
    assert np.array_equal(host(h), kept)
    assert np.array_equal(host(q), oq)
    assert np.array_equal(onv.unswizzle_sf(host(sf), rows, cols // 16), osf)


@contextlib.contextmanager
def _tiles(nv, mode):
    nv.nvfp4_set_gemm_tiles(mode)
    try:
        yield
    finally:
        nv.nvfp4_set_gemm_tiles(nv.GEMM_TILES_AUTO)


def test_compact_swiglu_bf16_epilogue_both_kernels(nv):
    sizes, counts, N, K = [512, 128, 384], [500, 128, 300], 512, 768
    rows_max = sum(sizes)
    G = len(sizes)
    a_q, a_sf = inputs.random_nvfp4_operand(92, 0, rows_max, K)
    b = [inputs.random_nvfp4_operand(92, 1 + g, N, K) for g in range(G)]

    def swz(sf_lin):
        r, k = sf_lin.shape
        out = torch.empty(nv.sf_bytes(r, 16 * k), dtype=torch.uint8, device="cuda")
        nv.nvfp4_sf_swizzle(dev(sf_lin), r, k, k, 1, out)
        return out

    a_q_d, a_sf_d = dev(a_q), swz(a_sf)
    b_q_d = dev(np.stack([x[0] for x in b]))
    b_sf_d = torch.stack([swz(x[1]) for x in b])
    offs_np = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    outs = {}
    for mode in ("single", "pair"):
        out = torch.full((rows_max, N // 2), 12288.0, dtype=torch.bfloat16, device="cuda")
        with _tiles(nv, {"single": nv.GEMM_TILES_SINGLE, "pair": nv.GEMM_TILES_PAIR}[mode]):
            nv.nvfp4_grouped_gemm(a_q_d, a_sf_d, rows_max, dev(offs_np), dev(np.array(counts, np.int32)), G, N, K,
                                  b_q_d, b_sf_d, 0.75, nv.EPI_SWIGLU_BF16, out_bf16=out)
        nv.nvfp4_device_status()
        outs[mode] = out.float().cpu().numpy()
    assert np.array_equal(outs["single"], outs["pair"])
    got = outs["single"]
    valid = np.concatenate([np.arange(offs_np[g], offs_np[g] + counts[g]) for g in range(G)])
    a_deq = onv.dequantize_rows(a_q, a_sf)
    b_deq = np.stack([onv.dequantize_rows(*x) for x in b])
    ref = omoe.l1_swiglu_bf16(omoe.grouped_gemm(a_deq, offs_np, b_deq, 0.75))
    assert rel_frobenius(got[valid].astype(np.float64), ref[valid]) <= 2e-3
    assert np.mean(got[valid] == ref[valid]) > 0.97
    mask = np.ones(rows_max, bool)
    mask[valid] = False
    assert np.all(got[mask] == 12288.0)
