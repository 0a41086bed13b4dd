"""GPU checks of the side combine: the combine of an earlier batch, run by two
extra warps of the CTA-pair L1 GEMM (or, with any other kernel, as its own
launch before it).

* y equals moe_combine's bit for bit (the same fp32 slot-order sum and one
  rounding), and the GEMM's own outputs are the bytes it writes without the
  side job, on both tile kernels, for short and long batches and top-k up to 32;
* a two-batch pipelined forward (batch 1's L1 runs batch 0's combine) gives
  each batch the y of the plain forward, bit for bit.
"""
import contextlib

import numpy as np
import pytest
import torch

import inputs
from oracle import moe as omoe

from gpu_util import built_lib, dev, host, rel_frobenius

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    built_lib()
    import nvfp4_block_scaled_moe_gb300 as nv
    from nvfp4_block_scaled_moe_gb300 import pipeline
    return nv, pipeline


@contextlib.contextmanager
def _tiles(nv, mode):
    nv.nvfp4_set_gemm_tiles(mode)
    try:
        yield
    finally:
        nv.nvfp4_set_gemm_tiles(nv.GEMM_TILES_AUTO)


def _swizzled(nv, sf_lin):
    rows, k_sf = sf_lin.shape
    out = torch.empty(nv.sf_bytes(rows, 16 * k_sf), dtype=torch.uint8, device="cuda")
    nv.nvfp4_sf_swizzle(dev(sf_lin), rows, k_sf, k_sf, 1, out)
    return out


@pytest.mark.parametrize("T,H,k", [(300, 1024, 8), (4100, 512, 4), (33, 7168, 32), (1, 64, 1)])
def test_side_combine_equals_combine(nv, T, H, k):
    nv, _ = nv
    sizes, counts, N, K = [512, 384, 256], [500, 300, 256], 512, 768
    rows_max, G = sum(sizes), len(sizes)
    a_q, a_sf = inputs.random_nvfp4_operand(61, 0, rows_max, K)
    b = [inputs.random_nvfp4_operand(61, 1 + g, N, K) for g in range(G)]
    a_q_d, a_sf_d = dev(a_q), _swizzled(nv, a_sf)
    b_q_d, b_sf_d = dev(np.stack([x[0] for x in b])), torch.stack([_swizzled(nv, x[1]) for x in b])
    offs = dev(np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32))
    cnt = dev(np.array(counts, np.int32))
    # the earlier batch: random BF16 rows, a permutation, weights
    rng = np.random.default_rng(T * H + k)
    n_rows = T * k + 5
    rows = dev(omoe.round_to_bf16(rng.standard_normal((n_rows, H))).astype(np.float32), torch.bfloat16)
    inv = dev(rng.permutation(n_rows)[:T * k].reshape(T, k).astype(np.int32))
    w = dev(rng.random((T, k)).astype(np.float32))
    y_ref = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    nv.moe_combine(rows, inv, w, y_ref)

    def gemm(side):
        oq = torch.full((rows_max, N // 4), 0x77, dtype=torch.uint8, device="cuda")
        osf = torch.zeros(nv.sf_bytes(rows_max, N // 2), dtype=torch.uint8, device="cuda")
        y = torch.full((T, H), 7.0, dtype=torch.bfloat16, device="cuda")
        nv.nvfp4_grouped_gemm(a_q_d, a_sf_d, rows_max, offs, cnt, G, N, K, b_q_d, b_sf_d, 1.0, nv.EPI_SWIGLU_NVFP4,
                              out_q=oq, out_sf=osf, side_combine=(rows, inv, w, y) if side else None)
        nv.nvfp4_device_status()
        return host(oq), host(osf), y

    plain_q, plain_sf, _ = gemm(False)
    for mode in (nv.GEMM_TILES_PAIR, nv.GEMM_TILES_SINGLE):
        with _tiles(nv, mode):
            q, sf, y = gemm(True)
        assert np.array_equal(q, plain_q) and np.array_equal(sf, plain_sf)
        assert torch.equal(y, y_ref), mode


def test_pipelined_forward_equals_plain(nv):
    """Batch 1's L1 GEMM runs batch 0's combine; then batch 1's own combine.
    Both ys equal the plain forward's, and are within the oracle bound."""
    nv, pipeline = nv
    spec = inputs.moe_spec(T=600, H=1024, I=512, E=16, top_k=4, seed=62, zipf=True)
    s = pipeline.MoeShape(T=spec["T"], H=spec["H"], I=spec["I"], E=spec["E"], top_k=spec["top_k"])
    w = pipeline.MoeWeights(s)
    pool, o1, o2 = inputs.moe_weight_pool(spec)
    w.set_from_pool(torch.from_numpy(pool).cuda(), o1, o2, float(inputs.WEIGHT_STD))
    x_t, x = inputs.moe_x(spec)
    logits = inputs.moe_logits(spec)
    xs = [x_t.cuda(), x_t.flip(0).contiguous().cuda()]                 # two different batches
    lgs = [dev(logits), dev(np.ascontiguousarray(logits[::-1]))]
    plain = [pipeline.moe_forward(xs[i], lgs[i], w, pipeline.MoeBuffers(s)).clone() for i in range(2)]
    bufs = [pipeline.MoeBuffers(s), pipeline.MoeBuffers(s)]
    pipeline.moe_forward_deferred(xs[0], lgs[0], w, bufs[0])
    pipeline.moe_forward_deferred(xs[1], lgs[1], w, bufs[1], prev=bufs[0])     # runs batch 0's combine
    pipeline.moe_combine_deferred(bufs[1])
    nv.nvfp4_device_status()
    assert torch.equal(bufs[0].y, plain[0]) and torch.equal(bufs[1].y, plain[1])
    w1, w2 = inputs.moe_all_weights(spec)
    ref = omoe.moe_ffn(x, logits, w1, w2, spec["top_k"])["y"]
    assert rel_frobenius(bufs[0].y.float().cpu().numpy(), ref) <= 2e-2
