"""The path's launches replayed from CUDA graphs give the same bytes as eager calls.

bench.py times the standalone quantiser and the dense GEMM by replaying captured
launches; these tests check that capture changes nothing: each output of a
replay is compared bit for bit with the same call made eagerly (the quantiser,
both GEMM tile kernels, and a whole MoE step of route -> L1 -> L2 -> combine).
"""
import contextlib

import numpy as np
import pytest
import torch

import inputs

from gpu_util import built_lib, dev, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    built_lib()
    import nvfp4_block_scaled_moe_gb300 as nv
    return nv


def _replayed(fn, outs):
    """Zero outs, run fn eagerly, snapshot; zero again, capture fn, replay twice;
    compare (regions a call leaves unwritten stay zero on both sides)."""
    for o in outs:
        o.zero_()
    fn()
    torch.cuda.synchronize()
    eager = [o.clone() for o in outs]
    for o in outs:
        o.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fn()
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, outs):
        assert torch.equal(a, b)


def test_quantize_swiglu_in_graph(nv):
    rows, cols = 1024, 2048
    g = torch.Generator(device="cuda").manual_seed(5)
    gu = (torch.randn((rows, 2 * cols), generator=g, device="cuda") * 3).to(torch.bfloat16)
    q = torch.empty((rows, cols // 2), dtype=torch.uint8, device="cuda")
    sf = torch.empty(nv.sf_bytes(rows, cols), dtype=torch.uint8, device="cuda")
    _replayed(lambda: nv.nvfp4_quantize(gu, cols, nv.MODE_SWIGLU_GU8, q, sf), [q, sf])
    nv.nvfp4_device_status()


@contextlib.contextmanager
def _tiles(nv, mode):
    nv.nvfp4_set_gemm_tiles(mode)
    try:
        yield
    finally:
        nv.nvfp4_set_gemm_tiles(nv.GEMM_TILES_AUTO)


@pytest.mark.parametrize("mode", ["single", "pair", "auto"])
def test_grouped_gemm_in_graph(nv, mode):
    sizes, counts, N, K = [512, 128, 384], [500, 128, 300], 1024, 768
    rows_max = sum(sizes)
    a_q, a_sf = inputs.random_nvfp4_operand(71, 0, rows_max, K)
    b = [inputs.random_nvfp4_operand(71, 1 + g, N, K) for g in range(len(sizes))]

    def swz(sf_lin):
        r, k = sf_lin.shape
        out = torch.empty(nv.sf_bytes(r, 16 * k), dtype=torch.uint8, device="cuda")
        nv.nvfp4_sf_swizzle(dev(sf_lin), r, k, k, 1, out)
        return out

    a_q_d, a_sf_d = dev(a_q), swz(a_sf)
    b_q_d = dev(np.stack([x[0] for x in b]))
    b_sf_d = torch.stack([swz(x[1]) for x in b])
    offs = dev(np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32))
    cnt = dev(np.array(counts, np.int32))
    out = torch.zeros((rows_max, N), dtype=torch.bfloat16, device="cuda")
    oq = torch.zeros((rows_max, N // 4), dtype=torch.uint8, device="cuda")
    osf = torch.zeros(nv.sf_bytes(rows_max, N // 2), dtype=torch.uint8, device="cuda")

    def run():
        nv.nvfp4_grouped_gemm(a_q_d, a_sf_d, rows_max, offs, cnt, len(sizes), N, K, b_q_d, b_sf_d, 1.0,
                              nv.EPI_BF16, out_bf16=out)
        nv.nvfp4_grouped_gemm(a_q_d, a_sf_d, rows_max, offs, cnt, len(sizes), N, K, b_q_d, b_sf_d, 1.0,
                              nv.EPI_SWIGLU_NVFP4, out_q=oq, out_sf=osf)

    # auto: CTA pairs split with a single-CTA launch on a second stream (forked
    # and joined inside the captured call)
    with _tiles(nv, {"single": nv.GEMM_TILES_SINGLE, "pair": nv.GEMM_TILES_PAIR, "auto": nv.GEMM_TILES_AUTO}[mode]):
        _replayed(run, [out, oq, osf])
    nv.nvfp4_device_status()


def test_whole_moe_step_in_graph(nv):
    from nvfp4_block_scaled_moe_gb300 import pipeline
    spec = inputs.moe_spec(T=600, H=1024, I=512, E=16, top_k=4, seed=73, zipf=True)
    s = pipeline.MoeShape(T=spec["T"], H=spec["H"], I=spec["I"], E=spec["E"], top_k=spec["top_k"])
    w = pipeline.MoeWeights(s)
    pool, o1, o2 = inputs.moe_weight_pool(spec)
    w.set_from_pool(torch.from_numpy(pool).cuda(), o1, o2, float(inputs.WEIGHT_STD))
    b = pipeline.MoeBuffers(s)
    x_t, _ = inputs.moe_x(spec)
    x = x_t.cuda()
    logits = dev(inputs.moe_logits(spec))
    _replayed(lambda: pipeline.moe_forward(x, logits, w, b),
              [b.y, b.topk_ids, b.offsets, b.perm_token, b.inv_perm])
    nv.nvfp4_device_status()
    assert host(b.offsets)[-1] > 0
