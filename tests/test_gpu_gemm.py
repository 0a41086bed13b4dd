"""GPU parity: nvfp4_grouped_gemm (tcgen05 block-scaled MMA) against the oracle's
float64 GEMM on dequantised operands.

Operands are random packed E2M1 bytes with random (non-uniform) E4M3 scales
straight from the seeded generator; the device swizzles its own copy of the
scales with nvfp4_sf_swizzle, so nothing the oracle computes reaches the GPU.
Bounds: BF16 rows and SwiGLU h within relative Frobenius 2e-3 (and nearly all
BF16 values identical); re-quantised nibbles within the 0.1% / one-step bound.
Every case runs on both tile kernels (single CTAs with 128-row tiles, CTA pairs
with 256-row tiles where N % 256 == 0); each must meet the bounds, and the two
must agree bit for bit (same per-element K order of the same MMAs).
"""
import contextlib

import numpy as np
import pytest
import torch

import inputs
from oracle import moe as omoe
from oracle import nvfp4 as onv

from gpu_util import built_lib, compare_requantised, dev, host, rel_frobenius

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    built_lib()
    import nvfp4_block_scaled_moe_gb300 as nv
    return nv


def _swizzled(nv, sf_lin):
    rows, k_sf = sf_lin.shape
    out = torch.empty(nv.sf_bytes(rows, 16 * k_sf), dtype=torch.uint8, device="cuda")
    nv.nvfp4_sf_swizzle(dev(sf_lin), rows, k_sf, k_sf, 1, out)
    return out


def _operands(nv, seed, rows_max, group_sizes, N, K, sf_range=(0x30, 0x44)):
    a_q, a_sf = inputs.random_nvfp4_operand(seed, 0, rows_max, K, *sf_range)
    G = len(group_sizes)
    bq, bsf = zip(*(inputs.random_nvfp4_operand(seed, 1 + g, N, K, *sf_range) for g in range(G)))
    b_q, b_sf = np.stack(bq), np.stack(bsf)
    d = dict(a_q=dev(a_q), a_sf=_swizzled(nv, a_sf), b_q=dev(b_q),
             b_sf=torch.stack([_swizzled(nv, b_sf[g]) for g in range(G)]))
    offs = np.concatenate([[0], np.cumsum(group_sizes)]).astype(np.int32)
    a_deq = onv.dequantize_rows(a_q, a_sf)
    b_deq = np.stack([onv.dequantize_rows(b_q[g], b_sf[g]) for g in range(G)])
    return d, offs, a_deq, b_deq


@contextlib.contextmanager
def _tiles(nv, mode):
    nv.nvfp4_set_gemm_tiles(mode)
    try:
        yield
    finally:
        nv.nvfp4_set_gemm_tiles(nv.GEMM_TILES_AUTO)


def _both_kernels(nv, run):
    """run() -> tuple of host arrays, on each tile kernel (single CTAs and CTA
    pairs) and with the automatic choice (which splits a grouped pair GEMM's
    odd groups' last blocks off to a single-CTA launch beside it); asserts they
    are identical."""
    outs = []
    for mode in (nv.GEMM_TILES_SINGLE, nv.GEMM_TILES_PAIR, nv.GEMM_TILES_AUTO):
        with _tiles(nv, mode):
            outs.append(run())
    for o in outs[1:]:
        for a, b in zip(outs[0], o):
            assert np.array_equal(a, b), "the tile kernels differ"
    return outs[0]


def _valid_rows(offs, counts):
    rows = []
    for g in range(len(offs) - 1):
        rows.extend(range(offs[g], offs[g] + counts[g]))
    return np.array(rows, dtype=np.int64)


CASES_BF16 = [
    # (group padded sizes, counts or None, N, K, alpha)
    ([128], None, 128, 256, 1.0),                     # one tile, one K stage
    ([256], None, 512, 512, 1.0),
    ([384], None, 384, 1024, 1.0),                    # odd number of 128-column tiles
    ([128, 0, 384, 128], [100, 0, 300, 128], 768, 768, 0.75),
    ([128] * 40, [128 - (i % 7) for i in range(40)], 1024, 1280, 1.0),   # > one wave of tiles
    ([1024, 384, 640], [1024, 383, 600], 1792, 768, 1.0),                 # pairs, odd tails, > one wave
    # more groups than the CTA-pair kernel takes (single-CTA kernel), a third of them empty
    ([0 if i % 3 == 0 else 128 for i in range(600)], [0 if i % 3 == 0 else 1 + (i * 37) % 128 for i in range(600)],
     256, 256, 1.0),
    # long K: the epilogue's store spacing reaches its 320-cycle cap
    ([512, 256], [512, 250], 512, 2048, 1.0),
    ([256], None, 256, 4096, 0.5),
]


@pytest.mark.parametrize("sizes,counts,N,K,alpha", CASES_BF16)
def test_gemm_bf16_epilogue(nv, sizes, counts, N, K, alpha):
    rows_max = sum(sizes) + 128
    d, offs, a_deq, b_deq = _operands(nv, 11 + N + K, rows_max, sizes, N, K)

    def run():
        out = torch.full((rows_max, N), 12288.0, dtype=torch.bfloat16, device="cuda")
        if counts is None:
            nv.nvfp4_grouped_gemm(d["a_q"], d["a_sf"], sizes[0], None, None, 1, N, K, d["b_q"], d["b_sf"], alpha,
                                  nv.EPI_BF16, out_bf16=out)
        else:
            nv.nvfp4_grouped_gemm(d["a_q"], d["a_sf"], rows_max, dev(offs), dev(np.array(counts, np.int32)),
                                  len(sizes), N, K, d["b_q"], d["b_sf"], alpha, nv.EPI_BF16, out_bf16=out)
        nv.nvfp4_device_status()
        return (out.float().cpu().numpy(),)

    assert counts is not None or len(sizes) == 1
    valid = np.arange(sizes[0]) if counts is None else _valid_rows(offs, counts)
    (got,) = _both_kernels(nv, run)
    ref = omoe.round_to_bf16(omoe.grouped_gemm(a_deq[:offs[-1]], offs, b_deq, alpha))
    assert rel_frobenius(got[valid], ref[valid]) <= 2e-3
    assert np.mean(got[valid] == ref[valid]) > 0.97
    mask = np.ones(rows_max, bool)
    mask[valid] = False
    assert np.all(got[mask] == 12288.0)               # nothing stored outside the real rows


@pytest.mark.parametrize("epi", ["bf16", "swiglu"])
def test_split_gemm_equals_pair_and_single(nv, epi):
    """A grouped pair GEMM with many odd groups (auto tiles: the pair launch on
    all but eight SMs skips the half-empty pair tiles of the thinnest odd
    groups, which a single-CTA launch on those eight SMs computes beside it)
    gives the bytes of the pair kernel alone and of the single-CTA kernel
    alone, and the oracle's values."""
    blocks = [1, 3, 2, 0, 5, 1, 1, 4, 7, 1, 2, 3, 1, 0, 1, 9, 1, 1, 3, 1, 2, 1, 1, 6]   # 15 odd groups
    sizes = [128 * b for b in blocks]
    counts = [max(0, s - (i * 29) % 128) for i, s in enumerate(sizes)]
    rows_max = sum(sizes)
    assert rows_max >= 2 * 128 * len(sizes)            # the automatic choice takes CTA pairs
    N, K = 512, 512
    d, offs, a_deq, b_deq = _operands(nv, 91, rows_max, sizes, N, K)
    cnt = dev(np.array(counts, np.int32))

    def run():
        if epi == "bf16":
            out = torch.full((rows_max, N), 12288.0, dtype=torch.bfloat16, device="cuda")
            nv.nvfp4_grouped_gemm(d["a_q"], d["a_sf"], rows_max, dev(offs), cnt, len(sizes), N, K, d["b_q"],
                                  d["b_sf"], 1.0, nv.EPI_BF16, out_bf16=out)
            nv.nvfp4_device_status()
            return (out.float().cpu().numpy(),)
        q = torch.full((rows_max, N // 4), 0x77, dtype=torch.uint8, device="cuda")
        sf = torch.zeros(nv.sf_bytes(rows_max, N // 2), dtype=torch.uint8, device="cuda")
        nv.nvfp4_grouped_gemm(d["a_q"], d["a_sf"], rows_max, dev(offs), cnt, len(sizes), N, K, d["b_q"], d["b_sf"],
                              1.0, nv.EPI_SWIGLU_NVFP4, out_q=q, out_sf=sf)
        nv.nvfp4_device_status()
        return host(q), host(sf)

    outs = _both_kernels(nv, run)
    valid = _valid_rows(offs, counts)
    g_full = omoe.grouped_gemm(a_deq, offs, b_deq, 1.0)
    if epi == "bf16":
        ref = omoe.round_to_bf16(g_full)
        assert rel_frobenius(outs[0][valid], ref[valid]) <= 2e-3
    else:
        oq, osf, _ = omoe.l1_swiglu_requant(g_full)
        gsf = onv.unswizzle_sf(outs[1], rows_max, N // 32)
        res = compare_requantised(outs[0][valid], gsf[valid], oq[valid], osf[valid])
        assert res["ok"], res


CASES_SWIGLU = [
    ([128], None, 256, 256, 1.0),
    ([256, 128], [200, 128], 512, 1024, 1.25),
    ([128, 128, 0, 256], [1, 128, 0, 129], 256, 512, 0.5),
    ([768, 384, 128], [768, 300, 127], 1024, 512, 1.0),
]


@pytest.mark.parametrize("sizes,counts,N,K,alpha", CASES_SWIGLU)
def test_gemm_swiglu_nvfp4_epilogue(nv, sizes, counts, N, K, alpha):
    rows_max = sum(sizes)
    d, offs, a_deq, b_deq = _operands(nv, 7 + N + K, rows_max, sizes, N, K)
    I = N // 2

    def run(with_h):
        q = torch.full((rows_max, I // 2), 0x77, dtype=torch.uint8, device="cuda")
        sf = torch.zeros(nv.sf_bytes(rows_max, I), dtype=torch.uint8, device="cuda")
        h = torch.zeros((rows_max, I), dtype=torch.float32, device="cuda") if with_h else None
        if counts is None:
            nv.nvfp4_grouped_gemm(d["a_q"], d["a_sf"], rows_max, None, None, 1, N, K, d["b_q"], d["b_sf"], alpha,
                                  nv.EPI_SWIGLU_NVFP4, out_q=q, out_sf=sf, h_debug=h)
        else:
            nv.nvfp4_grouped_gemm(d["a_q"], d["a_sf"], rows_max, dev(offs), dev(np.array(counts, np.int32)),
                                  len(sizes), N, K, d["b_q"], d["b_sf"], alpha, nv.EPI_SWIGLU_NVFP4, out_q=q,
                                  out_sf=sf, h_debug=h)
        nv.nvfp4_device_status()
        return (host(q), host(sf)) + ((host(h),) if with_h else ())

    valid = np.arange(rows_max) if counts is None else _valid_rows(offs, counts)
    gq, gsf_sw, gh = _both_kernels(nv, lambda: run(True))
    nq, nsf, = _both_kernels(nv, lambda: run(False))          # the h_debug stores change nothing else
    assert np.array_equal(nq, gq) and np.array_equal(nsf, gsf_sw)
    g_full = omoe.grouped_gemm(a_deq, offs, b_deq, alpha)
    oq, osf, oh = omoe.l1_swiglu_requant(g_full)
    assert rel_frobenius(gh[valid], oh[valid]) <= 2e-3
    gsf = onv.unswizzle_sf(gsf_sw, rows_max, I // 16)
    res = compare_requantised(gq[valid], gsf[valid], oq[valid], osf[valid])
    assert res["ok"], res
    untouched = np.ones(rows_max, bool)
    untouched[valid] = False
    assert np.all(gq[untouched] == 0x77)


def test_gemm_uniform_vs_random_scales_both_match(nv):
    """All-equal scales hide a wrong scale layout; random ones expose it.  Both must match."""
    for sf_range in ((0x38, 0x38), (0x28, 0x50)):
        d, offs, a_deq, b_deq = _operands(nv, 3, 256, [256], 256, 512, sf_range)

        def run():
            out = torch.empty((256, 256), dtype=torch.bfloat16, device="cuda")
            nv.nvfp4_grouped_gemm(d["a_q"], d["a_sf"], 256, None, None, 1, 256, 512, d["b_q"], d["b_sf"], 1.0,
                                  nv.EPI_BF16, out_bf16=out)
            return (out.float().cpu().numpy(),)

        (got,) = _both_kernels(nv, run)
        ref = omoe.round_to_bf16(omoe.grouped_gemm(a_deq, offs, b_deq))
        assert rel_frobenius(got, ref) <= 2e-3, sf_range


def test_gemm_one_hot_locates_nibbles_and_scales(nv):
    """A single nonzero A element at (r, k) and a single nonzero B element at (n, k):
    the product appears only at (r, n), scaled by both blocks' scales."""
    K, N, M = 512, 256, 256
    rng = np.random.default_rng(9)
    for r, n, k in ((0, 0, 0), (5, 77, 37), (127, 255, 511), (64, 3, 300), (33, 200, 64), (100, 128, 130),
                    (128, 0, 0), (200, 255, 17), (255, 129, 480)):                 # rows of the odd CTA
        a_q = np.zeros((M, K // 2), np.uint8)
        b_q = np.zeros((1, N, K // 2), np.uint8)
        a_q[r, k // 2] = (0x3 << 4) if k % 2 else 0x3          # 1.5
        b_q[0, n, k // 2] = (0x6 << 4) if k % 2 else 0x6       # 4.0
        a_sf = rng.integers(0x30, 0x40, (M, K // 16), dtype=np.uint8)
        b_sf = rng.integers(0x30, 0x40, (N, K // 16), dtype=np.uint8)

        def run():
            out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
            nv.nvfp4_grouped_gemm(dev(a_q), _swizzled(nv, a_sf), M, None, None, 1, N, K, dev(b_q),
                                  _swizzled(nv, b_sf)[None], 1.0, nv.EPI_BF16, out_bf16=out)
            return (out.float().cpu().numpy(),)

        (got,) = _both_kernels(nv, run)
        expect = np.zeros((M, N))
        expect[r, n] = 1.5 * 4.0 * onv.e4m3_decode(a_sf[r, k // 16]) * onv.e4m3_decode(b_sf[n, k // 16])
        assert np.array_equal(got, omoe.round_to_bf16(expect)), (r, n, k)


def test_dense_config_full_size_sampled_rows(nv):
    """The dense L1 workload at full size (8192 x 4096 x 7168, seeded as bench.py
    runs it, the same launch: tile kernel by default, SwiGLU + NVFP4 epilogue).
    The GPU-quantised operands are bit-exact (all of B, sampled rows of A); on
    sampled output rows h matches the float64 GEMM of the dequantised operands,
    the re-quantised codes stay within the bound, and they are bit-exact against
    the oracle fed the kernel's own h.  Without h_debug the bytes are the same."""
    spec = dict(inputs.CONFIGS["dense"])
    M, N, K = spec["M"], spec["N"], spec["K"]
    I = N // 2
    a, bw = inputs.dense_inputs(spec)
    a_d, b_d = torch.from_numpy(a).cuda(), torch.from_numpy(bw).cuda()
    a_q = torch.empty((M, K // 2), dtype=torch.uint8, device="cuda")
    a_sf = torch.empty(nv.sf_bytes(M, K), dtype=torch.uint8, device="cuda")
    b_q = torch.empty((N, K // 2), dtype=torch.uint8, device="cuda")
    b_sf = torch.empty(nv.sf_bytes(N, K), dtype=torch.uint8, device="cuda")
    nv.nvfp4_quantize(a_d, K, nv.MODE_PLAIN, a_q, a_sf)
    nv.nvfp4_quantize(b_d, K, nv.MODE_PLAIN, b_q, b_sf)
    out_q = torch.empty((M, I // 2), dtype=torch.uint8, device="cuda")
    out_sf = torch.empty(nv.sf_bytes(M, I), dtype=torch.uint8, device="cuda")
    h = torch.empty((M, I), dtype=torch.float32, device="cuda")
    nv.nvfp4_grouped_gemm(a_q, a_sf, M, None, None, 1, N, K, b_q, b_sf[None], 1.0, nv.EPI_SWIGLU_NVFP4,
                          out_q=out_q, out_sf=out_sf, h_debug=h)
    q2, sf2 = torch.empty_like(out_q), torch.empty_like(out_sf)
    nv.nvfp4_grouped_gemm(a_q, a_sf, M, None, None, 1, N, K, b_q, b_sf[None], 1.0, nv.EPI_SWIGLU_NVFP4,
                          out_q=q2, out_sf=sf2)
    nv.nvfp4_device_status()
    assert torch.equal(out_q, q2) and torch.equal(out_sf, sf2)
    ob_q, ob_sf = onv.quantize_rows(bw)
    assert np.array_equal(host(b_q), ob_q)
    assert np.array_equal(onv.unswizzle_sf(host(b_sf), N, K // 16), ob_sf)
    # random rows, and the last row of every 128-row band (the edge of each tile's A block)
    pick = np.unique(np.concatenate([np.random.default_rng(12).choice(M, 22, replace=False), [0, M - 1],
                                     np.arange(127, M, 128)]))
    oa_q, oa_sf = onv.quantize_rows(a[pick])
    assert np.array_equal(host(a_q)[pick], oa_q)
    assert np.array_equal(onv.unswizzle_sf(host(a_sf), M, K // 16)[pick], oa_sf)
    g = onv.dequantize_rows(oa_q, oa_sf) @ onv.dequantize_rows(ob_q, ob_sf).T
    oq, osf, oh = omoe.l1_swiglu_requant(g)
    gh = host(h)[pick]
    assert rel_frobenius(gh, oh) <= 2e-3
    gq = host(out_q)[pick]
    gsf = onv.unswizzle_sf(host(out_sf), M, I // 16)[pick]
    res = compare_requantised(gq, gsf, oq, osf)
    assert res["ok"], res
    hq, hsf = onv.quantize_rows(gh)
    assert np.array_equal(hq, gq) and np.array_equal(hsf, gsf)


def test_dense_l2_shape_full_size_sampled_rows(nv):
    """The L2-shaped dense workload at full size (16384 x 7168 x 2048, BF16 rows,
    seeded as bench.py runs it, the same launch): every tile spaces its epilogue
    stores at the 320-cycle cap.  On sampled output rows (the first, the last and
    rows of 32-row slices at tile edges) the BF16 rows match the float64 GEMM of
    the oracle-quantised operands, rounded once to BF16; a second launch writes
    the same bytes."""
    spec = dict(inputs.CONFIGS["dense_l2"])
    M, N, K = spec["M"], spec["N"], spec["K"]
    a, bw = inputs.dense_inputs(spec)
    a_d, b_d = torch.from_numpy(a).cuda(), torch.from_numpy(bw).cuda()
    a_q = torch.empty((M, K // 2), dtype=torch.uint8, device="cuda")
    a_sf = torch.empty(nv.sf_bytes(M, K), dtype=torch.uint8, device="cuda")
    b_q = torch.empty((N, K // 2), dtype=torch.uint8, device="cuda")
    b_sf = torch.empty(nv.sf_bytes(N, K), dtype=torch.uint8, device="cuda")
    nv.nvfp4_quantize(a_d, K, nv.MODE_PLAIN, a_q, a_sf)
    nv.nvfp4_quantize(b_d, K, nv.MODE_PLAIN, b_q, b_sf)
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    out2 = torch.empty_like(out)
    for o in (out, out2):
        nv.nvfp4_grouped_gemm(a_q, a_sf, M, None, None, 1, N, K, b_q, b_sf[None], 1.0, nv.EPI_BF16, out_bf16=o)
    nv.nvfp4_device_status()
    assert torch.equal(out, out2)
    ob_q, ob_sf = onv.quantize_rows(bw)
    assert np.array_equal(host(b_q), ob_q)
    edges = [255, 256, 8191, 8192, 16128 + 31, 16128 + 32]
    pick = np.unique(np.concatenate([np.random.default_rng(13).choice(M, 16, replace=False), [0, M - 1], edges]))
    oa_q, oa_sf = onv.quantize_rows(a[pick])
    assert np.array_equal(host(a_q)[pick], oa_q)
    ref = omoe.round_to_bf16(onv.dequantize_rows(oa_q, oa_sf) @ onv.dequantize_rows(ob_q, ob_sf).T)
    got = out.float().cpu().numpy()[pick]
    assert rel_frobenius(got, ref) <= 2e-3
    assert np.mean(got == ref) > 0.97
